"""Brute-force float64 model of the KVBuffer algorithm for one (request, value head).

Test helper only.  It restates, token by token and without any batching, the
buffered computation that the library's kernels perform, so that the CPU tests
can check the algebra of the buffered form against the recurrent oracle (the
exactness claim of "KVBuffer: IO-aware Serving for Linear Attention",
"Core claim" and "What would settle it" sections):

* decode with n buffered tokens since the last flush (state S0), current token t:
      A_i = a_1 + ... + a_i  (cumulative log-gate since the flush, i = 1..n+1)
      pseudo-value  u_t = v_t                                    (plain / gated)
                    u_t = beta_t (v_t - e^{A_t} S0^T k_t
                                  - sum_{i<=n} e^{A_t-A_i} (k_t.k_i) u_i)   (gated delta)
      o_t = e^{A_t} S0^T q_t + sum_{i<=n+1} e^{A_t-A_i} (q_t.k_i) u_i
* flush of L buffered tokens (Figure 1: the state is updated with all buffered
  KVs and written back to its slot):
      S <- e^{A_L} S0 + sum_{i<=L} e^{A_L-A_i} k_i u_i^T
* verify T drafts: the decode formula applied to each draft in turn, each
  draft appended to the buffer, the state untouched (Figure 2);
  accept(j): keep the first j drafts; flush all if the buffer holds >= m.
* a draft tree: each draft sees the committed buffer plus its ancestors only;
  accepting a node keeps its path from the root.

It shares no code with the oracle or the library.
"""
from __future__ import annotations

import numpy as np

PLAIN, GATED, GATED_DELTA = 0, 1, 2


class BufferedHead:
    def __init__(self, S0, variant, m, scale=1.0):
        self.S = np.array(S0, dtype=np.float64)
        self.variant = variant
        self.m = m
        self.scale = scale
        self.buf = []  # entries: dict(k, u, a)
        self.flushes = 0

    def _token_out(self, q, k, v, a, b):
        """Output and pseudo-value of one token appended after the current buffer."""
        q = np.asarray(q, dtype=np.float64) * self.scale
        k = np.asarray(k, dtype=np.float64)
        v = np.asarray(v, dtype=np.float64)
        a = 0.0 if a is None else float(a)
        A_prev = [0.0]
        for e in self.buf:
            A_prev.append(A_prev[-1] + e["a"])
        A = A_prev[1:]  # cumulative of buffered tokens
        A_t = A_prev[-1] + a
        if self.variant == GATED_DELTA:
            corr = np.exp(A_t) * (self.S.T @ k)
            for e, Ai in zip(self.buf, A):
                corr = corr + np.exp(A_t - Ai) * float(k @ e["k"]) * e["u"]
            u = float(b) * (v - corr)
        else:
            u = v
        o = np.exp(A_t) * (self.S.T @ q)
        for e, Ai in zip(self.buf, A):
            o = o + np.exp(A_t - Ai) * float(q @ e["k"]) * e["u"]
        o = o + float(q @ k) * u
        return o, {"k": k, "u": u, "a": a}

    def flush(self):
        A = np.cumsum([e["a"] for e in self.buf]) if self.buf else np.zeros(0)
        if not self.buf:
            return
        A_L = A[-1]
        S = np.exp(A_L) * self.S
        for e, Ai in zip(self.buf, A):
            S = S + np.exp(A_L - Ai) * np.outer(e["k"], e["u"])
        self.S = S
        self.buf = []
        self.flushes += 1

    def decode(self, q, k, v, a=None, b=None, auto_flush=True):
        o, entry = self._token_out(q, k, v, a, b)
        self.buf.append(entry)
        if auto_flush and len(self.buf) == self.m:
            self.flush()
        return o

    def verify(self, drafts):
        """drafts: list of (q, k, v, a, b).  Appends all drafts; returns their outputs."""
        outs = []
        for (q, k, v, a, b) in drafts:
            o, entry = self._token_out(q, k, v, a, b)
            self.buf.append(entry)
            outs.append(o)
        self._pending = len(drafts)
        return np.array(outs)

    def accept(self, j):
        T = self._pending
        n = len(self.buf) - T
        self.buf = self.buf[: n + j]
        if len(self.buf) >= self.m:
            self.flush()

    def verify_tree(self, drafts, parents):
        """Draft tree: draft j sees the committed buffer plus its ancestors' entries
        in path order (parents[j] < j, -1 for a child of the last accepted token).
        The committed buffer is unchanged; returns the drafts' outputs."""
        base = list(self.buf)
        entries, outs = [], []
        for j, (q, k, v, a, b) in enumerate(drafts):
            anc, p = [], parents[j]
            while p >= 0:
                anc.append(p)
                p = parents[p]
            self.buf = base + [entries[i] for i in reversed(anc)]
            o, entry = self._token_out(q, k, v, a, b)
            entries.append(entry)
            outs.append(o)
        self.buf = base
        self._tree = (entries, list(parents))
        return np.array(outs)

    def accept_path(self, node):
        """Keep the path from the root to draft ``node`` (-1: none); flush at >= m."""
        entries, parents = self._tree
        path, p = [], node
        while p >= 0:
            path.append(p)
            p = parents[p]
        self.buf = self.buf + [entries[i] for i in reversed(path)]
        if len(self.buf) >= self.m:
            self.flush()

    def current_state(self):
        """The full recurrent state (flushed state plus the buffered tokens folded in)."""
        saved_S, saved_buf, saved_f = self.S.copy(), list(self.buf), self.flushes
        self.flush()
        S = self.S
        self.S, self.buf, self.flushes = saved_S, saved_buf, saved_f
        return S
