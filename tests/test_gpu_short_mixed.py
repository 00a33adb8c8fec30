"""GPU parity: mixed ragged batch of short-context (buffer-only) and long requests.

Workload: the scalar-gated layer (16 heads, d=128, bf16), B=512 rows per step:
256 short-context requests, each with a total length drawn from U{1..64},
served from a 64-slot buffer (8 blocks of 8) with no state, retired when done
and replaced by a fresh request with new random blocks; 256 long requests
with a state and an initial buffer occupancy drawn from U{0..7}, m = 8, one
8-slot block each; blocks come from a shared pool of 4096 with random block
tables.  256 steps, each one kvb_decode launch for the long rows and one
kvb_short_ctx launch for the short rows.  Lengths are compared bit for bit
for every request each step; outputs for sampled requests (and every
incarnation of the sampled short slots) against the oracle (the recurrence
from S = 0 for short requests).
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

    long_sample = [3, 77, 200]
    short_sample = [int(short_ids[0]), int(short_ids[100]), int(short_ids[255])]
    long_hist = {r: {k_: [] for k_ in ("q", "k", "v", "log_g")} for r in long_sample}
    for r in long_sample:
        for k_ in long_hist[r]:
            long_hist[r][k_].extend(list(wtok[k_][:occ[r], r]))
    long_out = {r: [] for r in long_sample}
    short_hist = {r: {k_: [] for k_ in ("q", "k", "v", "log_g")} for r in short_sample}
    short_out = {r: [] for r in short_sample}
    short_done = []  # (history, outputs) of finished incarnations
    tol = tol_for(layer)

    for t in range(steps):
        lt = I.draw_tokens(rng, layer, (n_long,))
        st = I.draw_tokens(rng, layer, (n_short,))
        o_l = pool.decode(long_ids, *token_tensors(lt, layer, slice(None)))
        o_s = pool.short_ctx(short_ids, *token_tensors(st, layer, slice(None)))
        n_model[:n_long] += 1
        n_model[:n_long][n_model[:n_long] >= m] = 0
        n_model[n_long:] += 1
        ol, osh = o_l.cpu().numpy(), o_s.cpu().numpy()
        for r in long_sample:
            for k_ in long_hist[r]:
                long_hist[r][k_].append(lt[k_][r])
            long_out[r].append(ol[r])
        for r in short_sample:
            i = r - n_long
            for k_ in short_hist[r]:
                short_hist[r][k_].append(st[k_][i])
            short_out[r].append(osh[i])
        assert np.array_equal(pool.get_lengths(), n_model.astype(np.int32)), t
        # retire finished short requests and admit fresh ones in their place
        for r in short_ids:
            r = int(r)
            if n_model[r] == short_len[r]:
                if r in short_sample:
                    short_done.append((short_hist[r], short_out[r]))
                    short_hist[r] = {k_: [] for k_ in ("q", "k", "v", "log_g")}
                    short_out[r] = []
                pool.release_request(r)
                free[:0] = owned[r]  # released blocks go back to the pool
                n_model[r] = 0
                short_len[r] = int(rng.integers(1, 65))
                owned[r] = [int(free.pop()) for _ in range(short_blocks)]
                pool.set_request(r, -1, owned[r])

    for r in long_sample:
        hist = {k_: np.stack(v_) for k_, v_ in long_hist[r].items()}
        hist["beta"] = None
        o_ref, _, _ = oracle.decode_sequence(S0[r], hist, layer.variant)
        assert rel_err(np.stack(long_out[r]), o_ref[occ[r]:]) <= tol, r
    for r in short_sample:
        if short_out[r]:
            short_done.append((short_hist[r], short_out[r]))
    for hist_l, outs in short_done:
        hist = {k_: np.stack(v_) for k_, v_ in hist_l.items()}
        hist["beta"] = None
        o_ref = oracle.short_context(hist, layer.variant, layer.d_k, layer.d_v)
        assert rel_err(np.stack(outs), o_ref) <= tol
    assert len(short_done) >= 6
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())
    assert pool.get_error() is None

