"""fp64 CPU oracle for KV-buffered linear-attention decoding.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
baseline / reference arm import this module.  The library's product path never
calls it, and it shares no code with the CUDA kernels or their host library.

What it computes
----------------
KVBuffer ("KVBuffer: IO-aware Serving for Linear Attention", abstract and the
"Core claim" / "Load-bearing premise" sections of its summary page) changes
*when* the linear-attention state is updated and *how often it crosses
memory*, and claims the outputs are exactly those of the ordinary per-token
recurrence.  So the oracle is that per-token recurrence, written out plainly in
float64, with no buffer, no chunking and no flush threshold.  The page's
"What would settle it" section proposes exactly this comparison: run the same
tokens through the recurrent form and the buffered form and check the outputs
match.

The pages print no equation (the referee report's minor comment notes that the
update rule is never written down), so the recurrences are the standard ones of
the works the page cites:

* plain linear attention (Katharopoulos et al., reference [6]):
      S_t = S_{t-1} + k_t v_t^T
* scalar-gated linear attention (gated linear attention [20], Mamba-2/SSD [2]):
      S_t = g_t S_{t-1} + k_t v_t^T,          g_t = exp(a_t)
* gated delta rule (Gated DeltaNet [19], DeltaNet [21]):
      S_t = g_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
* output, after the current token's update:
      o_t = scale * S_t^T q_t

S is d_k x d_v per (request, value head); o = S^T q (the GDN paper writes the
transposed orientation; the result is the same).  A value head h uses the
query/key head h // (H_v / H_k) (contiguous grouping; the pages are silent).

Speculative verification and accept (Figure 2 of the page): every draft's
output is the recurrent output with the earlier drafts in the history, and the
state after accepting a prefix of j drafts is the recurrent state after those j
tokens.  Short-context decoding (abstract: outputs computed directly from
buffered keys and values, without creating the state) is the recurrence from
S = 0.  A tree of drafts is verified node by node along each node's path from
the root, and accepting a node keeps exactly that path.

Parity status: every function here is pinned by tests that do not reuse this
code (closed forms, exact rational arithmetic, reductions between variants, the
delta rule as a gradient step computed by autograd, the chunked UT form solved
with a library solver, and brute force); see tests/test_oracle_pins.py.
"""
from __future__ import annotations

import numpy as np

PLAIN, GATED, GATED_DELTA = 0, 1, 2


def _f64(x):
    return None if x is None else np.asarray(x, dtype=np.float64)


def expand_qk(x, n_v_heads: int):
    """Map query/key heads onto value heads: value head h reads q/k head h // (Hv/Hk).

    ``x`` has the head axis second to last: [..., Hk, d].  Returns [..., Hv, d].
    """
    x = _f64(x)
    hk = x.shape[-2]
    if n_v_heads % hk != 0:
        raise ValueError("n_v_heads must be a multiple of n_qk_heads")
    return np.repeat(x, n_v_heads // hk, axis=-2)


def recurrent_step(S, q, k, v, log_g, beta, variant: int, scale: float = 1.0):
    """One token of the recurrent form.

    S: [..., d_k, d_v] float64 (not modified).  q, k: [..., d_k] (already mapped
    onto value heads), v: [..., d_v], log_g, beta: [...] or None.
    Returns (S_t, o_t) with o_t = scale * S_t^T q.
    """
    S = _f64(S)
    q, k, v = _f64(q), _f64(k), _f64(v)
    outer_kv = k[..., :, None] * v[..., None, :]
    if variant == PLAIN:
        S_new = S + outer_kv
    elif variant == GATED:
        g = np.exp(_f64(log_g))[..., None, None]
        S_new = g * S + outer_kv
    elif variant == GATED_DELTA:
        g = np.ones(S.shape[:-2]) if log_g is None else np.exp(_f64(log_g))
        b = _f64(beta)
        # (I - beta k k^T) S = S - beta k (k^T S)
        kTS = np.einsum("...i,...ij->...j", k, S)
        erased = S - b[..., None, None] * (k[..., :, None] * kTS[..., None, :])
        S_new = g[..., None, None] * erased + b[..., None, None] * outer_kv
    else:
        raise ValueError(f"unknown variant {variant}")
    o = scale * np.einsum("...ij,...i->...j", S_new, q)
    return S_new, o


def recurrent_scan(S0, q, k, v, log_g=None, beta=None, variant: int = PLAIN,
                   scale: float = 1.0, keep_states=()):
    """Run the recurrence over tokens along axis 0.

    S0: [..., d_k, d_v]; q, k: [T, ..., Hk, d_k] with the head axis second to
    last (they are mapped onto value heads here); v: [T, ..., Hv, d_v];
    log_g, beta: [T, ..., Hv] or None.  S0's leading axes must match
    v's [..., Hv].  Returns (o [T, ..., Hv, d_v], S_T, {t: S_t for t in keep_states})
    where S_t is the state after token index t (0-based).
    """
    S = _f64(S0).copy()
    v = _f64(v)
    n_tok = v.shape[0]
    hv = v.shape[-2]
    qe = expand_qk(q, hv)
    ke = expand_qk(k, hv)
    out = np.empty(v.shape, dtype=np.float64)
    kept = {}
    keep = set(int(t) for t in keep_states)
    for t in range(n_tok):
        lg = None if log_g is None else log_g[t]
        bt = None if beta is None else beta[t]
        S, out[t] = recurrent_step(S, qe[t], ke[t], v[t], lg, bt, variant, scale)
        if t in keep:
            kept[t] = S.copy()
    return out, S, kept


def decode_sequence(S0, tokens: dict, variant: int, scale: float = 1.0, keep_states=()):
    """Decode a token sequence from state S0 (the oracle of every decode step).

    ``tokens`` holds q, k, v, log_g, beta laid out [T, ...] as in recurrent_scan.
    """
    return recurrent_scan(S0, tokens["q"], tokens["k"], tokens["v"], tokens.get("log_g"),
                          tokens.get("beta"), variant, scale, keep_states)


def verify(S_pre, drafts: dict, variant: int, scale: float = 1.0):
    """Outputs of T draft tokens verified against the pre-round state.

    Draft j's output is the recurrent output after the history plus drafts
    0..j (Figure 2: the same result the baseline gets from its temporary state
    j).  The state itself is not advanced.  Returns o: [T, ..., Hv, d_v].
    """
    o, _, _ = decode_sequence(S_pre, drafts, variant, scale)
    return o


def accept(S_pre, drafts: dict, n_accepted, variant: int, scale: float = 1.0):
    """State after accepting the first ``n_accepted`` drafts of each request.

    S_pre: [B, Hv, d_k, d_v]; drafts laid out [T, B, ...]; n_accepted: [B]
    integers in [0, T].  Request r's state is the recurrent replay of its
    first n_accepted[r] drafts only (rejected drafts leave no trace).
    """
    S_pre = _f64(S_pre)
    n_acc = np.asarray(n_accepted)
    S_out = S_pre.copy()
    for r in range(S_pre.shape[0]):
        j = int(n_acc[r])
        if j == 0:
            continue
        sub = {key: (None if val is None else val[:j, r]) for key, val in drafts.items()}
        _, S_r, _ = decode_sequence(S_pre[r], sub, variant, scale)
        S_out[r] = S_r
    return S_out


def tree_path(parents, j: int):
    """Draft indices on the path from the root to draft j, root first.

    parents[i] is the draft that draft i continues (-1: it continues the last
    accepted token), always an earlier index.
    """
    path = []
    while j >= 0:
        path.append(int(j))
        j = int(parents[j])
    return path[::-1]


def verify_tree(S_pre, drafts: dict, parents, variant: int, scale: float = 1.0):
    """Outputs of a tree of T drafts verified against the pre-round state.

    Tree-shaped speculation (the draft trees the page cites for speculative
    decoding): draft j's output is the recurrent output after the history plus
    the drafts on the path from the root to j, in path order.  drafts laid out
    [T, ...] as in decode_sequence; returns o: [T, ..., Hv, d_v].  A chain
    (parents[j] = j - 1) is ordinary verification.
    """
    T = drafts["v"].shape[0]
    o = np.empty(drafts["v"].shape, dtype=np.float64)
    for j in range(T):
        path = tree_path(parents, j)
        sub = {key: (None if val is None else val[path]) for key, val in drafts.items()}
        o_path, _, _ = decode_sequence(S_pre, sub, variant, scale)
        o[j] = o_path[-1]
    return o


def accept_tree(S_pre, drafts: dict, parents, node: int, variant: int, scale: float = 1.0):
    """State after accepting the path from the root to draft ``node`` (-1: none)."""
    if node < 0:
        return _f64(S_pre).copy()
    path = tree_path(parents, node)
    sub = {key: (None if val is None else val[path]) for key, val in drafts.items()}
    _, S, _ = decode_sequence(S_pre, sub, variant, scale)
    return S


def short_context(tokens: dict, variant: int, d_k: int, d_v: int, scale: float = 1.0):
    """Outputs of a request that never builds a state: the recurrence from S = 0.

    tokens laid out [T, Hk|Hv, d]; returns o: [T, Hv, d_v].
    """
    hv = tokens["v"].shape[-2]
    S0 = np.zeros((hv, d_k, d_v))
    o, _, _ = decode_sequence(S0, tokens, variant, scale)
    return o


def prefill_state(tokens: dict, variant: int, d_k: int, d_v: int, lead_shape: tuple):
    """State after a prompt, starting from S = 0 (the recurrence, token by token).

    tokens laid out [T, *lead_shape, H, d]; returns S: [*lead_shape, Hv, d_k, d_v].
    """
    hv = tokens["v"].shape[-2]
    S0 = np.zeros(tuple(lead_shape) + (hv, d_k, d_v))
    _, S, _ = decode_sequence(S0, tokens, variant)
    return S


def gated_prefill_closed_form(tokens: dict, variant: int):
    """State after a prompt from S = 0 for the plain and scalar-gated forms, unrolled.

    Unrolling S_t = g_t S_{t-1} + k_t v_t^T from S_0 = 0 gives
        S_T = sum_i (prod_{j > i} g_j) k_i v_i^T = K^T diag(w) V,
        w_i = exp(sum_{j > i} a_j),
    one matrix product per (request, head).  Used to build large prefill states
    quickly; pinned against ``prefill_state`` in the tests.
    tokens laid out [T, *lead, H, d]; returns [*lead, Hv, d_k, d_v].
    """
    if variant not in (PLAIN, GATED):
        raise ValueError("closed form exists only for the plain and gated variants")
    v = _f64(tokens["v"])
    hv = v.shape[-2]
    k = expand_qk(tokens["k"], hv)
    if variant == GATED:
        a = _f64(tokens["log_g"])  # [T, ..., Hv]
        suffix = np.cumsum(a[::-1], axis=0)[::-1]  # sum_{j >= i} a_j
        w = np.exp(suffix - a)  # sum_{j > i} a_j
    else:
        w = np.ones(v.shape[:-1])
    kw = k * w[..., None]
    # move token axis last for a batched matmul: [..., d_k, T] @ [..., T, d_v]
    kw_t = np.moveaxis(kw, 0, -1)
    v_t = np.moveaxis(v, 0, -2)
    return kw_t @ v_t
