"""GPU parity: mixed ragged batch of short-context (buffer-only) and long requests.

Workload: the scalar-gated layer (16 heads, d=128, bf16), B=512 rows per step:
256 short-context requests, each with a total length drawn from U{1..64},
served from a 64-slot buffer (8 blocks of 8) with no state, retired when done
and replaced by a fresh request with new random blocks; 256 long requests
with a state and an initial buffer occupancy drawn from U{0..7}, m = 8, one
8-slot block each; blocks come from a shared pool of 4096 with random block
tables.  256 steps, each one kvb_decode launch for the long rows and one
kvb_short_ctx launch for the short rows.  Lengths are compared bit for bit
for every request each step; the output of every request at every step
against the oracle (the recurrence over the request's whole history, from
S = 0 for every incarnation of a short request), per tensor.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests import oracle_pool
from tests.gpu_harness import make_pool, token_tensors, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def test_mixed_short_long():
    w = I.WORKLOADS["mixed_B512_gated"]
    layer, m, bs = w.layer, w.m, w.block_size
    n_short = w.extra["n_short"]
    n_long = w.batch - n_short
    short_blocks = w.extra["short_cap"] // bs
    num_blocks = w.extra["num_blocks"]
    steps = w.steps
    rng = np.random.default_rng(w.seed)
    pool = make_pool(layer, m, w.batch, short_blocks, bs, num_blocks=num_blocks,
                     num_slots=n_long, max_blocks=short_blocks)
    free = list(rng.permutation(num_blocks))
    long_ids = np.arange(n_long)
    short_ids = np.arange(n_long, w.batch)
    S0 = I.draw_state(rng, layer, n_long)
    pool.state.copy_(torch.from_numpy(S0))
    for r in long_ids:
        pool.set_request(int(r), int(r), [int(free.pop())])
    short_len, owned = {}, {}
    for r in short_ids:
        owned[int(r)] = [int(free.pop()) for _ in range(short_blocks)]
        pool.set_request(int(r), -1, owned[int(r)])
        short_len[int(r)] = int(rng.integers(1, 65))

    # long requests start with U{0..7} buffered tokens (decoded on subsets: ragged launches)
    occ = rng.integers(0, m, size=n_long)
    wtok = I.draw_tokens(rng, layer, (m - 1, n_long))
    for s in range(m - 1):
        rows = np.nonzero(occ > s)[0]
        if len(rows):
            pool.decode(rows, *token_tensors(wtok, layer, (s, rows)))
    n_model = np.zeros(w.batch, dtype=np.int64)
    n_model[:n_long] = occ
    assert np.array_equal(pool.get_lengths(), n_model)

    lt_all = []  # every step's long-request tokens
    st_all = []  # every step's short-request tokens
    out_l = np.empty((steps, n_long, layer.n_v_heads, layer.d_v), dtype=np.float32)
    out_s = np.empty((steps, n_short, layer.n_v_heads, layer.d_v), dtype=np.float32)
    start = np.zeros(n_short, dtype=np.int64)  # step at which each short slot's incarnation began
    incarnations = []  # (slot, first step, last step + 1)

    for t in range(steps):
        lt = I.draw_tokens(rng, layer, (n_long,))
        st = I.draw_tokens(rng, layer, (n_short,))
        lt_all.append(lt)
        st_all.append(st)
        out_l[t] = pool.decode(long_ids, *token_tensors(lt, layer, slice(None))).cpu().numpy()
        out_s[t] = pool.short_ctx(short_ids, *token_tensors(st, layer, slice(None))).cpu().numpy()
        n_model[:n_long] += 1
        n_model[:n_long][n_model[:n_long] >= m] = 0
        n_model[n_long:] += 1
        assert np.array_equal(pool.get_lengths(), n_model.astype(np.int32)), t
        # retire finished short requests and admit fresh ones in their place
        for r in short_ids:
            r = int(r)
            if n_model[r] == short_len[r]:
                i = r - n_long
                incarnations.append((i, int(start[i]), t + 1))
                start[i] = t + 1
                pool.release_request(r)
                free[:0] = owned[r]  # released blocks go back to the pool
                n_model[r] = 0
                short_len[r] = int(rng.integers(1, 65))
                owned[r] = [int(free.pop()) for _ in range(short_blocks)]
                pool.set_request(r, -1, owned[r])
    for i in range(n_short):  # unfinished incarnations are compared too
        if start[i] < steps:
            incarnations.append((i, int(start[i]), steps))
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())
    assert pool.get_error() is None
    torch.cuda.synchronize()
    states = pool.state.cpu().numpy()

    def stack(tok_list, key):
        return None if tok_list[0][key] is None else np.stack([x[key] for x in tok_list])

    L = {key: stack(lt_all, key) for key in ("q", "k", "v", "log_g", "beta")}  # [steps, n_long, ...]
    Sx = {key: stack(st_all, key) for key in ("q", "k", "v", "log_g", "beta")}

    # long requests: one oracle task per chunk with the same warm-up length
    tasks = []
    for o in np.unique(occ):
        same = np.nonzero(occ == o)[0]
        for part in np.array_split(same, max(1, len(same) // 8)):
            hist = {key: (None if val is None else
                          np.concatenate([wtok[key][:o, part], val[:, part]]))
                    for key, val in L.items()}
            n_tot = int(o) + steps
            tasks.append(dict(S0=S0[part], hist=hist, out=out_l[:, part], state=states[part],
                              fold_at=np.full(len(part), n_tot - n_tot % m - 1),
                              variant=layer.variant, rows=part))
    res = oracle_pool.run(oracle_pool.decode_errors, tasks)
    err_long = np.zeros(n_long)
    err_state = np.zeros(n_long)
    for task, (eo, es) in zip(tasks, res):
        err_long[task["rows"]] = eo
        err_state[task["rows"]] = es
    tol = tol_for(layer)
    assert err_long.max() <= tol, (err_long.max(), int(err_long.argmax()))
    assert err_state.max() <= tol, (err_state.max(), int(err_state.argmax()))

    # short requests: every incarnation is the recurrence from S = 0 over its own tokens
    items = []
    for i, t0, t1 in incarnations:
        hist = {key: (None if val is None else val[t0:t1, i]) for key, val in Sx.items()}
        items.append((hist, out_s[t0:t1, i]))
    assert len(items) >= n_short
    groups = [items[g::32] for g in range(32)]
    res = oracle_pool.run(oracle_pool.short_errors,
                          [dict(items=g, variant=layer.variant, d_k=layer.d_k, d_v=layer.d_v)
                           for g in groups if g])
    err_short = np.concatenate(res)
    assert err_short.max() <= tol, err_short.max()
