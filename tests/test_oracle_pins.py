"""Pins for the fp64 oracle: checks against facts that do not come from the oracle itself.

Each pin is a function of the oracle module so that ``test_planted_mistakes``
can re-run all of them against deliberately broken copies of the recurrence
(a planted mistake must make at least one pin fail).

What pins what:
* plain recurrence       closed form o_t = S0^T q_t + sum_{i<=t} (q_t.k_i) v_i (loops),
                         exact rational arithmetic on integer inputs, hand-worked fixture
* scalar-gated           constant-gate closed form, product-of-gates brute force,
                         g == 1 reduces to plain bit for bit
* gated delta rule       beta = 0 is pure decay; beta = 1 with unit k stores v exactly
                         (S_t^T k_t = v_t); one step equals a gradient step on
                         1/2 ||S^T k - v||^2 computed by torch autograd; a whole chunk
                         equals the UT-transform chunk form solved by numpy.linalg.solve
* buffered form          the KVBuffer algorithm (brute-force model) equals the oracle
                         for every flush threshold m <= 6, every variant
* verify / accept        accept(j) equals the replay of j tokens; j = 0 keeps the state
* draft trees            exact rationals along each root path (plain), constant-gate path
                         weights (order), chain = verify, star = single decodes, and the
                         buffered algorithm with an ancestor mask
* short context          equals the closed form from S = 0
* GQA mapping            value head h reads q/k head h // (Hv/Hk)
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
from oracle import kvb_oracle
from tests.buffered_model import BufferedHead

PLAIN, GATED, GATED_DELTA = oracle.PLAIN, oracle.GATED, oracle.GATED_DELTA
HERE = os.path.dirname(os.path.abspath(__file__))


def _rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def _tokens(rng, T, B, hk, hv, dk, dv, variant, unit_k=False):
    q = _rand(rng, T, B, hk, dk, scale=0.5)
    k = _rand(rng, T, B, hk, dk, scale=0.5)
    if unit_k:
        k = k / np.linalg.norm(k, axis=-1, keepdims=True)
    v = _rand(rng, T, B, hv, dv)
    lg = None if variant == PLAIN else rng.uniform(-0.3, 0.0, size=(T, B, hv))
    beta = rng.uniform(0.05, 0.95, size=(T, B, hv)) if variant == GATED_DELTA else None
    return {"q": q, "k": k, "v": v, "log_g": lg, "beta": beta}


# --------------------------------------------------------------------------- pins
def pin_plain_closed_form(orc):
    rng = np.random.default_rng(11)
    T, dk, dv = 9, 5, 3
    S0 = _rand(rng, dk, dv)
    q, k, v = _rand(rng, T, 1, dk), _rand(rng, T, 1, dk), _rand(rng, T, 1, dv)
    o, S_T, _ = orc.recurrent_scan(S0[None], q, k, v, variant=PLAIN)
    for t in range(T):
        for c in range(dv):
            ref = sum(S0[i, c] * q[t, 0, i] for i in range(dk))
            for s in range(t + 1):
                ref += sum(q[t, 0, i] * k[s, 0, i] for i in range(dk)) * v[s, 0, c]
            assert abs(o[t, 0, c] - ref) <= 1e-12 * (1 + abs(ref)), (t, c)
    S_ref = S0 + sum(np.outer(k[s, 0], v[s, 0]) for s in range(T))
    assert np.abs(S_T[0] - S_ref).max() <= 1e-12


def pin_plain_exact_rational(orc):
    rng = np.random.default_rng(12)
    T, dk, dv = 7, 2, 3
    qi = rng.integers(-3, 4, size=(T, 1, dk))
    ki = rng.integers(-3, 4, size=(T, 1, dk))
    vi = rng.integers(-3, 4, size=(T, 1, dv))
    S0i = rng.integers(-3, 4, size=(1, dk, dv))
    o, S_T, _ = orc.recurrent_scan(S0i.astype(float), qi.astype(float), ki.astype(float),
                                   vi.astype(float), variant=PLAIN)
    S = [[Fraction(int(S0i[0, i, c])) for c in range(dv)] for i in range(dk)]
    for t in range(T):
        for i in range(dk):
            for c in range(dv):
                S[i][c] += Fraction(int(ki[t, 0, i])) * Fraction(int(vi[t, 0, c]))
        for c in range(dv):
            exact = sum(S[i][c] * Fraction(int(qi[t, 0, i])) for i in range(dk))
            assert o[t, 0, c] == float(exact)
    for i in range(dk):
        for c in range(dv):
            assert S_T[0, i, c] == float(S[i][c])


def pin_scale_exact_rational(orc):
    """The output scale multiplies the output once: o_t = s * S_t^T q_t, exactly.

    Integer inputs and s = 3/8 make every oracle value an exact binary fraction,
    so the oracle must agree bit for bit with rational arithmetic.  s = 3/8 is
    not a power of two and not 1, so applying it twice (9/64), not at all, or to
    the state update instead of the output, all differ from the exact value.
    """
    rng = np.random.default_rng(16)
    T, dk, dv = 6, 3, 2
    s = Fraction(3, 8)
    qi = rng.integers(-3, 4, size=(T, 1, dk))
    ki = rng.integers(-3, 4, size=(T, 1, dk))
    vi = rng.integers(-3, 4, size=(T, 1, dv))
    S0i = rng.integers(-3, 4, size=(1, dk, dv))
    o, S_T, _ = orc.recurrent_scan(S0i.astype(float), qi.astype(float), ki.astype(float),
                                   vi.astype(float), variant=PLAIN, scale=float(s))
    S = [[Fraction(int(S0i[0, i, c])) for c in range(dv)] for i in range(dk)]
    for t in range(T):
        for i in range(dk):
            for c in range(dv):
                S[i][c] += Fraction(int(ki[t, 0, i])) * Fraction(int(vi[t, 0, c]))
        for c in range(dv):
            exact = s * sum(S[i][c] * Fraction(int(qi[t, 0, i])) for i in range(dk))
            assert o[t, 0, c] == float(exact), (t, c)
    for i in range(dk):
        for c in range(dv):
            assert S_T[0, i, c] == float(S[i][c])  # the state carries no scale
    # the delta rule with the same scale: s times the unscaled outputs, and the
    # same states (the scale touches only the output)
    tok = _tokens(rng, 5, 1, 1, 1, 4, 3, GATED_DELTA)
    S0 = _rand(rng, 1, 1, 4, 3)
    o1, S1, _ = orc.recurrent_scan(S0, tok["q"], tok["k"], tok["v"], tok["log_g"], tok["beta"],
                                   variant=GATED_DELTA)
    o2, S2, _ = orc.recurrent_scan(S0, tok["q"], tok["k"], tok["v"], tok["log_g"], tok["beta"],
                                   variant=GATED_DELTA, scale=0.375)
    assert np.array_equal(S1, S2)
    assert np.abs(o2 - 0.375 * o1).max() <= 1e-15 * max(1.0, np.abs(o1).max())


def pin_gated_constant_gate(orc):
    rng = np.random.default_rng(13)
    T, dk, dv = 10, 4, 3
    g = 0.8
    S0 = _rand(rng, 1, dk, dv)
    q, k, v = _rand(rng, T, 1, dk), _rand(rng, T, 1, dk), _rand(rng, T, 1, dv)
    lg = np.full((T, 1), np.log(g))
    o, _, _ = orc.recurrent_scan(S0, q, k, v, lg, variant=GATED)
    for t in range(T):
        ref = g ** (t + 1) * (S0[0].T @ q[t, 0])
        for s in range(t + 1):
            ref = ref + g ** (t - s) * (q[t, 0] @ k[s, 0]) * v[s, 0]
        assert np.abs(o[t, 0] - ref).max() <= 1e-12


def pin_gated_product_of_gates(orc):
    rng = np.random.default_rng(14)
    T, dk, dv = 8, 3, 4
    S0 = _rand(rng, 2, dk, dv)
    tok = _tokens(rng, T, 1, 2, 2, dk, dv, GATED)
    o, _, _ = orc.recurrent_scan(S0[None], tok["q"], tok["k"], tok["v"], tok["log_g"], variant=GATED)
    g = np.exp(tok["log_g"])
    for h in range(2):
        for t in range(T):
            decay0 = 1.0
            for j in range(t + 1):
                decay0 *= g[j, 0, h]
            ref = decay0 * (S0[h].T @ tok["q"][t, 0, h])
            for s in range(t + 1):
                d = 1.0
                for j in range(s + 1, t + 1):
                    d *= g[j, 0, h]
                ref = ref + d * (tok["q"][t, 0, h] @ tok["k"][s, 0, h]) * tok["v"][s, 0, h]
            assert np.abs(o[t, 0, h] - ref).max() <= 1e-12


def pin_gated_unit_gate_is_plain(orc):
    rng = np.random.default_rng(15)
    T = 6
    S0 = _rand(rng, 1, 2, 5, 4)
    tok = _tokens(rng, T, 1, 2, 2, 5, 4, PLAIN)
    o_p, S_p, _ = orc.recurrent_scan(S0, tok["q"], tok["k"], tok["v"], variant=PLAIN)
    o_g, S_g, _ = orc.recurrent_scan(S0, tok["q"], tok["k"], tok["v"], np.zeros((T, 1, 2)),
                                     variant=GATED)
    assert np.array_equal(o_p, o_g) and np.array_equal(S_p, S_g)


def pin_delta_beta_zero_decay(orc):
    rng = np.random.default_rng(16)
    T, dk, dv = 7, 4, 3
    S0 = _rand(rng, 1, 1, dk, dv)
    tok = _tokens(rng, T, 1, 1, 1, dk, dv, GATED_DELTA)
    tok["beta"] = np.zeros((T, 1, 1))
    o, S_T, _ = orc.recurrent_scan(S0, tok["q"], tok["k"], tok["v"], tok["log_g"], tok["beta"],
                                   variant=GATED_DELTA)
    decay = 1.0
    for t in range(T):
        decay *= np.exp(tok["log_g"][t, 0, 0])
        ref = decay * (S0[0, 0].T @ tok["q"][t, 0, 0])
        assert np.abs(o[t, 0, 0] - ref).max() <= 1e-12
    assert np.abs(S_T[0, 0] - decay * S0[0, 0]).max() <= 1e-12


def pin_delta_overwrite(orc):
    rng = np.random.default_rng(17)
    T, dk, dv = 6, 5, 3
    S = _rand(rng, 1, 1, dk, dv)
    tok = _tokens(rng, T, 1, 1, 1, dk, dv, GATED_DELTA, unit_k=True)
    tok["beta"] = np.ones((T, 1, 1))
    for t in range(T):
        S, _ = orc.recurrent_step(S, tok["q"][t], tok["k"][t], tok["v"][t], tok["log_g"][t],
                                  tok["beta"][t], GATED_DELTA)
        recalled = S[0, 0].T @ tok["k"][t, 0, 0]
        assert np.abs(recalled - tok["v"][t, 0, 0]).max() <= 1e-12


def pin_delta_gradient_step(orc):
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(18)
    dk, dv = 5, 4
    S = _rand(rng, dk, dv)
    for _ in range(5):
        q, k, v = _rand(rng, dk), _rand(rng, dk, scale=0.5), _rand(rng, dv)
        lg, beta = rng.uniform(-0.3, 0.0), rng.uniform(0.1, 0.9)
        S_dec = torch.tensor(np.exp(lg) * S, requires_grad=True)
        loss = 0.5 * ((S_dec.T @ torch.tensor(k) - torch.tensor(v)) ** 2).sum()
        loss.backward()
        S_ref = (S_dec - beta * S_dec.grad).detach().numpy()
        S_new, o = orc.recurrent_step(S[None], q[None], k[None], v[None], np.array([lg]),
                                      np.array([beta]), GATED_DELTA)
        assert np.abs(S_new[0] - S_ref).max() <= 1e-12
        assert np.abs(o[0] - S_ref.T @ q).max() <= 1e-12
        S = S_new[0]


def pin_delta_ut_chunk_form(orc):
    rng = np.random.default_rng(19)
    L, dk, dv = 9, 6, 4
    S0 = _rand(rng, dk, dv)
    tok = _tokens(rng, L, 1, 1, 1, dk, dv, GATED_DELTA)
    o, S_L, _ = orc.recurrent_scan(S0[None, None], tok["q"], tok["k"], tok["v"], tok["log_g"],
                                   tok["beta"], variant=GATED_DELTA)
    K, Q, V = tok["k"][:, 0, 0], tok["q"][:, 0, 0], tok["v"][:, 0, 0]
    a, b = tok["log_g"][:, 0, 0], tok["beta"][:, 0, 0]
    A = np.cumsum(a)
    Gam = np.exp(A[:, None] - A[None, :])
    M = np.eye(L) + np.tril(b[:, None] * Gam * (K @ K.T), -1)
    rhs = b[:, None] * (V - np.exp(A)[:, None] * (K @ S0))
    U = np.linalg.solve(M, rhs)
    S_ref = np.exp(A[-1]) * S0 + K.T @ (np.exp(A[-1] - A)[:, None] * U)
    O_ref = np.exp(A)[:, None] * (Q @ S0) + (np.tril(Gam) * (Q @ K.T)) @ U
    assert np.abs(S_L[0, 0] - S_ref).max() <= 1e-11
    assert np.abs(o[:, 0, 0] - O_ref).max() <= 1e-11


def _run_buffered_vs_oracle(orc, variant, m, T=20, seed=20):
    rng = np.random.default_rng(seed + 7 * m + variant)
    dk, dv = 4, 3
    S0 = _rand(rng, dk, dv)
    tok = _tokens(rng, T, 1, 1, 1, dk, dv, variant, unit_k=(variant == GATED_DELTA))
    o_ref, _, states = orc.recurrent_scan(S0[None, None], tok["q"], tok["k"], tok["v"],
                                          tok["log_g"], tok["beta"], variant=variant,
                                          keep_states=range(T))
    head = BufferedHead(S0, variant, m)
    for t in range(T):
        a = None if tok["log_g"] is None else tok["log_g"][t, 0, 0]
        b = None if tok["beta"] is None else tok["beta"][t, 0, 0]
        o = head.decode(tok["q"][t, 0, 0], tok["k"][t, 0, 0], tok["v"][t, 0, 0], a, b)
        assert np.abs(o - o_ref[t, 0, 0]).max() <= 1e-11, (variant, m, t)
        if not head.buf:  # just flushed: the stored state is the recurrent state
            assert np.abs(head.S - states[t][0, 0]).max() <= 1e-11
        assert np.abs(head.current_state() - states[t][0, 0]).max() <= 1e-11


def pin_buffered_equals_recurrent(orc):
    for variant in (PLAIN, GATED, GATED_DELTA):
        for m in range(1, 7):
            _run_buffered_vs_oracle(orc, variant, m)


def pin_verify_accept(orc):
    for variant in (GATED, GATED_DELTA):
        rng = np.random.default_rng(30 + variant)
        dk, dv, m = 4, 3, 4
        S0 = _rand(rng, dk, dv)
        head = BufferedHead(S0, variant, m)
        S_hist = S0[None, None].copy()
        for rnd in range(8):
            T = int(rng.integers(1, 5))
            tok = _tokens(rng, T, 1, 1, 1, dk, dv, variant, unit_k=(variant == GATED_DELTA))
            o_orc = orc.verify(S_hist, tok, variant)
            drafts = [(tok["q"][t, 0, 0], tok["k"][t, 0, 0], tok["v"][t, 0, 0],
                       None if tok["log_g"] is None else tok["log_g"][t, 0, 0],
                       None if tok["beta"] is None else tok["beta"][t, 0, 0]) for t in range(T)]
            o_buf = head.verify(drafts)
            assert np.abs(o_buf - o_orc[:, 0, 0]).max() <= 1e-11
            j = int(rng.integers(0, T + 1))
            head.accept(j)
            S_new = orc.accept(S_hist, tok, np.array([j]), variant)
            if j == 0:
                assert np.array_equal(S_new, S_hist)
            # replay of exactly j tokens
            sub = {key: (None if val is None else val[:j]) for key, val in tok.items()}
            if j:
                _, S_rep, _ = orc.decode_sequence(S_hist, sub, variant)
                assert np.abs(S_new - S_rep).max() <= 1e-12
            S_hist = S_new
            assert np.abs(head.current_state() - S_hist[0, 0]).max() <= 1e-11


def pin_short_context(orc):
    rng = np.random.default_rng(40)
    T, dk, dv = 9, 4, 3
    tok = _tokens(rng, T, 1, 2, 2, dk, dv, PLAIN)
    tok = {key: (None if val is None else val[:, 0]) for key, val in tok.items()}
    o = orc.short_context(tok, PLAIN, dk, dv)
    for h in range(2):
        for t in range(T):
            ref = sum((tok["q"][t, h] @ tok["k"][s, h]) * tok["v"][s, h] for s in range(t + 1))
            assert np.abs(o[t, h] - ref).max() <= 1e-12
    for variant in (GATED, GATED_DELTA):
        tk = _tokens(rng, T, 1, 1, 1, dk, dv, variant, unit_k=True)
        tk1 = {key: (None if val is None else val[:, 0]) for key, val in tk.items()}
        o = orc.short_context(tk1, variant, dk, dv)
        head = BufferedHead(np.zeros((dk, dv)), variant, m=10 ** 9)
        for t in range(T):
            a = tk1["log_g"][t, 0]
            b = None if tk1["beta"] is None else tk1["beta"][t, 0]
            ob = head.decode(tk1["q"][t, 0], tk1["k"][t, 0], tk1["v"][t, 0], a, b)
            assert np.abs(ob - o[t, 0]).max() <= 1e-12


def pin_gqa_mapping(orc):
    rng = np.random.default_rng(50)
    T, dk, dv = 5, 3, 2
    hk, hv = 2, 4
    S0 = _rand(rng, 1, hv, dk, dv)
    tok = _tokens(rng, T, 1, hk, hv, dk, dv, GATED_DELTA)
    o, _, _ = orc.recurrent_scan(S0, tok["q"], tok["k"], tok["v"], tok["log_g"], tok["beta"],
                                 variant=GATED_DELTA)
    for h in range(hv):
        g = h // (hv // hk)
        single = {"q": tok["q"][:, :, g:g + 1], "k": tok["k"][:, :, g:g + 1],
                  "v": tok["v"][:, :, h:h + 1], "log_g": tok["log_g"][:, :, h:h + 1],
                  "beta": tok["beta"][:, :, h:h + 1]}
        o1, _, _ = orc.decode_sequence(S0[:, h:h + 1], single, GATED_DELTA)
        assert np.array_equal(o1[:, :, 0], o[:, :, h])
    # and the expansion itself: heads (0,1) read q/k head 0, heads (2,3) read head 1
    x = np.arange(2 * 3).reshape(2, 3).astype(float)
    assert np.array_equal(orc.expand_qk(x, 4), np.array([x[0], x[0], x[1], x[1]]))


def pin_gated_prefill_closed_form(orc):
    rng = np.random.default_rng(60)
    T = 30
    for variant in (PLAIN, GATED):
        tok = _tokens(rng, T, 2, 2, 2, 5, 4, variant)
        S_rec = orc.prefill_state(tok, variant, 5, 4, (2,))
        S_cf = orc.gated_prefill_closed_form(tok, variant)
        assert np.abs(S_rec - S_cf).max() <= 1e-12


def pin_hand_worked(orc):
    with open(os.path.join(HERE, "golden", "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        n = len(c["q"])
        lg = None if c["log_g"] is None else np.array(c["log_g"], dtype=float).reshape(n, 1, 1)
        bt = None if c["beta"] is None else np.array(c["beta"], dtype=float).reshape(n, 1, 1)
        o, S_T, _ = orc.recurrent_scan(np.array(c["S0"], dtype=float)[None, None],
                                       np.array(c["q"], dtype=float)[:, None, None],
                                       np.array(c["k"], dtype=float)[:, None, None],
                                       np.array(c["v"], dtype=float)[:, None, None],
                                       lg, bt, variant=c["variant"])
        assert np.abs(o[:, 0, 0] - np.array(c["o"])).max() <= 1e-12, c["name"]
        assert np.abs(S_T[0, 0] - np.array(c["S_final"])).max() <= 1e-12, c["name"]


TREE = [-1, 0, 0, 1, -1, 3, 2]  # two roots; draft 0 branches into 1 and 2; depth 4


def _walk(parents, j):
    nodes = []
    while j != -1:
        nodes.append(j)
        j = parents[j]
    return nodes[::-1]


def pin_tree_exact_rational(orc):
    """Draft trees, plain form on integers: draft j's output is q_j^T (S_pre + sum over
    its root path of k v^T), in exact rational arithmetic; constant gate g: the path
    weights g^(depth - position) fix the path order."""
    rng = np.random.default_rng(70)
    T, dk, dv = len(TREE), 3, 2
    S_pre = rng.integers(-3, 4, size=(dk, dv))
    q, k, v = (rng.integers(-3, 4, size=(T, d)) for d in (dk, dk, dv))
    drafts = {"q": q[:, None, :].astype(float), "k": k[:, None, :].astype(float),
              "v": v[:, None, :].astype(float), "log_g": None, "beta": None}
    o = orc.verify_tree(S_pre[None].astype(float), drafts, TREE, PLAIN)
    for j in range(T):
        S = [[Fraction(int(S_pre[a][c])) for c in range(dv)] for a in range(dk)]
        for i in _walk(TREE, j):
            for a in range(dk):
                for c in range(dv):
                    S[a][c] += int(k[i][a]) * int(v[i][c])
        exp = [sum(int(q[j][a]) * S[a][c] for a in range(dk)) for c in range(dv)]
        assert np.array_equal(o[j, 0], np.array([float(x) for x in exp])), j
    S_acc = orc.accept_tree(S_pre[None].astype(float), drafts, TREE, 5, PLAIN)
    exp = S_pre + sum(np.outer(k[i], v[i]) for i in (0, 1, 3, 5))
    assert np.array_equal(S_acc[0], exp.astype(float))
    assert np.array_equal(orc.accept_tree(S_pre[None].astype(float), drafts, TREE, -1, PLAIN)[0],
                          S_pre.astype(float))
    # constant gate: o_j = q_j^T (g^D S_pre + sum_p g^(D-p) k_(path p) v_(path p)^T)
    g = 0.7
    drafts_g = dict(drafts, log_g=np.full((T, 1), np.log(g)))
    og = orc.verify_tree(S_pre[None].astype(float), drafts_g, TREE, GATED)
    for j in range(T):
        path = _walk(TREE, j)
        D = len(path)
        S = g ** D * S_pre.astype(float)
        for pos, i in enumerate(path, start=1):
            S = S + g ** (D - pos) * np.outer(k[i], v[i])
        assert np.abs(og[j, 0] - S.T @ q[j]).max() <= 1e-12, j


def pin_tree_reductions(orc):
    """A chain tree is ordinary verification and accept; a star tree is T independent
    single-token decodes from the same state."""
    rng = np.random.default_rng(71)
    T = 5
    for variant in (PLAIN, GATED, GATED_DELTA):
        tok = _tokens(rng, T, 1, 1, 2, 4, 3, variant, unit_k=True)
        drafts = {key: (None if val is None else val[:, 0]) for key, val in tok.items()}
        S_pre = _rand(rng, 2, 4, 3)
        chain = list(range(-1, T - 1))
        assert np.abs(orc.verify_tree(S_pre, drafts, chain, variant)
                      - orc.verify(S_pre, drafts, variant)).max() <= 1e-12
        for j in range(T + 1):
            acc = orc.accept(S_pre[None], tok, np.array([j]), variant)[0]
            assert np.abs(orc.accept_tree(S_pre, drafts, chain, j - 1, variant) - acc).max() <= 1e-12
        star = [-1] * T
        o_star = orc.verify_tree(S_pre, drafts, star, variant)
        for j in range(T):
            one = {key: (None if val is None else val[j:j + 1]) for key, val in drafts.items()}
            o1, _, _ = orc.decode_sequence(S_pre, one, variant)
            assert np.abs(o_star[j] - o1[0]).max() <= 1e-12


def pin_buffered_tree_equals_recurrent(orc):
    """The buffered algorithm with an ancestor mask (committed buffer + the draft's path)
    equals the oracle's tree verification, and accepting a path equals its replay."""
    rng = np.random.default_rng(72)
    dk, dv = 4, 3
    for variant in (PLAIN, GATED, GATED_DELTA):
        for trial in range(4):
            m = 6
            S0 = _rand(rng, dk, dv)
            head = BufferedHead(S0, variant, m)
            S_hist = S0[None].copy()
            n0 = int(rng.integers(0, 3))
            pre = _tokens(rng, n0, 1, 1, 1, dk, dv, variant, unit_k=True)
            for t in range(n0):
                head.decode(pre["q"][t, 0, 0], pre["k"][t, 0, 0], pre["v"][t, 0, 0],
                            None if pre["log_g"] is None else pre["log_g"][t, 0, 0],
                            None if pre["beta"] is None else pre["beta"][t, 0, 0])
            if n0:
                _, S_hist, _ = orc.decode_sequence(
                    S_hist, {key: (None if val is None else val[:, 0]) for key, val in pre.items()},
                    variant)
            T = 6
            parents = [-1] + [int(rng.integers(-1, j)) for j in range(1, T)]
            tok = _tokens(rng, T, 1, 1, 1, dk, dv, variant, unit_k=True)
            drafts = {key: (None if val is None else val[:, 0]) for key, val in tok.items()}
            dl = [(tok["q"][t, 0, 0], tok["k"][t, 0, 0], tok["v"][t, 0, 0],
                   None if tok["log_g"] is None else tok["log_g"][t, 0, 0],
                   None if tok["beta"] is None else tok["beta"][t, 0, 0]) for t in range(T)]
            o = head.verify_tree(dl, parents)
            assert np.abs(o - orc.verify_tree(S_hist, drafts, parents, variant)[:, 0]).max() <= 1e-10
            node = int(rng.integers(-1, T))
            head.accept_path(node)
            S_acc = orc.accept_tree(S_hist, drafts, parents, node, variant)
            assert np.abs(head.current_state() - S_acc[0]).max() <= 1e-10


PINS = [pin_plain_closed_form, pin_plain_exact_rational, pin_scale_exact_rational,
        pin_gated_constant_gate,
        pin_gated_product_of_gates, pin_gated_unit_gate_is_plain, pin_delta_beta_zero_decay,
        pin_delta_overwrite, pin_delta_gradient_step, pin_delta_ut_chunk_form,
        pin_buffered_equals_recurrent, pin_verify_accept, pin_short_context, pin_gqa_mapping,
        pin_gated_prefill_closed_form, pin_hand_worked, pin_tree_exact_rational,
        pin_tree_reductions, pin_buffered_tree_equals_recurrent]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle)


# ------------------------------------------------------------------ planted mistakes
def _mut_gate_dropped(S, q, k, v, log_g, beta, variant, scale=1.0):
    if variant == GATED:
        log_g = np.zeros_like(np.asarray(log_g, dtype=float))
    return _ORIG_STEP(S, q, k, v, log_g, beta, variant, scale)


def _mut_erase_sign(S, q, k, v, log_g, beta, variant, scale=1.0):
    if variant != GATED_DELTA:
        return _ORIG_STEP(S, q, k, v, log_g, beta, variant, scale)
    S = np.asarray(S, float)
    k, v, q = np.asarray(k, float), np.asarray(v, float), np.asarray(q, float)
    g = np.exp(np.asarray(log_g, float))[..., None, None]
    b = np.asarray(beta, float)[..., None, None]
    kTS = np.einsum("...i,...ij->...j", k, S)
    S_new = g * (S + b * k[..., :, None] * kTS[..., None, :]) + b * k[..., :, None] * v[..., None, :]
    return S_new, scale * np.einsum("...ij,...i->...j", S_new, q)


def _mut_beta_missing_on_write(S, q, k, v, log_g, beta, variant, scale=1.0):
    if variant != GATED_DELTA:
        return _ORIG_STEP(S, q, k, v, log_g, beta, variant, scale)
    S = np.asarray(S, float)
    k, v, q = np.asarray(k, float), np.asarray(v, float), np.asarray(q, float)
    g = np.exp(np.asarray(log_g, float))[..., None, None]
    b = np.asarray(beta, float)[..., None, None]
    kTS = np.einsum("...i,...ij->...j", k, S)
    S_new = g * (S - b * k[..., :, None] * kTS[..., None, :]) + k[..., :, None] * v[..., None, :]
    return S_new, scale * np.einsum("...ij,...i->...j", S_new, q)


def _mut_output_before_update(S, q, k, v, log_g, beta, variant, scale=1.0):
    S_new, _ = _ORIG_STEP(S, q, k, v, log_g, beta, variant, scale)
    return S_new, scale * np.einsum("...ij,...i->...j", np.asarray(S, float), np.asarray(q, float))


def _mut_gate_after_write(S, q, k, v, log_g, beta, variant, scale=1.0):
    if variant != GATED:
        return _ORIG_STEP(S, q, k, v, log_g, beta, variant, scale)
    S = np.asarray(S, float)
    g = np.exp(np.asarray(log_g, float))[..., None, None]
    S_new = g * (S + np.asarray(k, float)[..., :, None] * np.asarray(v, float)[..., None, :])
    return S_new, scale * np.einsum("...ij,...i->...j", S_new, np.asarray(q, float))


def _mut_output_not_transposed(S, q, k, v, log_g, beta, variant, scale=1.0):
    S_new, _ = _ORIG_STEP(S, q, k, v, log_g, beta, variant, scale)
    qq = np.asarray(q, float)
    if S_new.shape[-1] != qq.shape[-1]:
        raise ValueError("shape mismatch")
    return S_new, scale * np.einsum("...ij,...j->...i", S_new, qq)


def _mut_scale_twice(S, q, k, v, log_g, beta, variant, scale=1.0):
    S_new, o = _ORIG_STEP(S, q, k, v, log_g, beta, variant, scale)
    return S_new, scale * o


def _mut_scale_dropped(S, q, k, v, log_g, beta, variant, scale=1.0):
    return _ORIG_STEP(S, q, k, v, log_g, beta, variant, 1.0)


def _mut_scale_on_key(S, q, k, v, log_g, beta, variant, scale=1.0):
    S_new, _ = _ORIG_STEP(S, q, scale * np.asarray(k, float), v, log_g, beta, variant, 1.0)
    return S_new, np.einsum("...ij,...i->...j", S_new, np.asarray(q, float))


def _mut_gqa_modulo(x, n_v_heads):
    x = np.asarray(x, float)
    hk = x.shape[-2]
    return np.concatenate([x] * (n_v_heads // hk), axis=-2)


def _mut_tree_path_without_node(parents, j):
    return _ORIG_TREE_PATH(parents, j)[:-1]


def _mut_tree_path_leaf_first(parents, j):
    return _ORIG_TREE_PATH(parents, j)[::-1]


_ORIG_STEP = kvb_oracle.recurrent_step
_ORIG_TREE_PATH = kvb_oracle.tree_path

MUTANTS = {
    "gate_dropped": ("recurrent_step", _mut_gate_dropped),
    "erase_sign": ("recurrent_step", _mut_erase_sign),
    "beta_missing_on_write": ("recurrent_step", _mut_beta_missing_on_write),
    "output_before_update": ("recurrent_step", _mut_output_before_update),
    "gate_after_write": ("recurrent_step", _mut_gate_after_write),
    "output_not_transposed": ("recurrent_step", _mut_output_not_transposed),
    "gqa_modulo": ("expand_qk", _mut_gqa_modulo),
    "scale_twice": ("recurrent_step", _mut_scale_twice),
    "scale_dropped": ("recurrent_step", _mut_scale_dropped),
    "scale_on_key": ("recurrent_step", _mut_scale_on_key),
    "tree_path_without_node": ("tree_path", _mut_tree_path_without_node),
    "tree_path_leaf_first": ("tree_path", _mut_tree_path_leaf_first),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistakes(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(kvb_oracle, attr, fn)
    failed = []
    for pin in PINS:
        try:
            pin(kvb_oracle)
        except Exception:  # an assertion or a shape error both count as caught
            failed.append(pin.__name__)
    assert failed, f"planted mistake {name!r} passed every pin"
