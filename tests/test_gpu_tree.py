"""GPU parity: verification of draft trees (kvb_verify_tree / kvb_accept_tree).

Each request gets its own random tree (parents[j] < j), on top of a committed
buffer of random length.  Every draft's output is compared with the fp64
oracle's recurrence along the draft's root path; after a random path is
accepted (often one that must be moved to the front of the draft slots), the
requests decode on and verify again, so a wrong compaction of keys, values,
pseudo-values or cumulative gates shows up in later outputs and states.
Lengths are compared bit for bit.  Covers the tensor-core verify (bf16,
d = 128), the FMA verify (fp32, d = 64 and 128) and batches split over several
launches.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import kvb_mod, make_pool, rel_err, token_tensors, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _row(tok, r):
    return {key: (None if val is None else val[r]) for key, val in tok.items()}


def _random_tree(rng, T):
    return [-1] + [int(rng.integers(-1, j)) for j in range(1, T)]


def _path(parents, j):
    out = []
    while j >= 0:
        out.append(j)
        j = parents[j]
    return out[::-1]


@pytest.mark.parametrize("layer,B", [
    (I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm"), 6),
    (I.Layer(I.GATED, 2, 2, 128, 128, "bf16"), 6),
    (I.Layer(I.GATED_DELTA, 1, 2, 64, 64, "f32", qk_dist="l2norm"), 6),
    (I.Layer(I.PLAIN, 1, 1, 128, 128, "f32"), 4),
    (I.Layer(I.GATED_DELTA, 1, 1, 64, 64, "bf16", qk_dist="l2norm"), 133),
], ids=["gated_delta_d128_bf16", "gated_d128_bf16", "gated_delta_d64_f32", "plain_d128_f32",
        "gated_delta_d64_bf16_B133"])
def test_tree_verify_accept_decode(layer, B):
    rng = np.random.default_rng(500 + B + layer.d_k + layer.variant)
    m, nb, bs = 8, 3, 8
    pool = make_pool(layer, m, B, nb, bs)
    S0 = I.draw_state(rng, layer, B)
    pool.state.copy_(torch.from_numpy(S0))
    perm = rng.permutation(B * nb)
    for r in range(B):
        pool.set_request(r, r, [int(x) for x in perm[r * nb:(r + 1) * nb]])
    S = [S0[r].astype(np.float64) for r in range(B)]
    n = np.zeros(B, dtype=np.int64)
    req = np.arange(B)
    tol = tol_for(layer)
    sample = range(B) if B <= 8 else list(range(0, B, 11)) + [B - 1]

    def decode_round():
        tok = I.draw_tokens(rng, layer, (B,))
        o = pool.decode(req, *token_tensors(tok, layer, slice(None))).cpu().numpy()
        for r in range(B):
            one = {key: (None if val is None else val[r:r + 1]) for key, val in tok.items()}
            o_ref, S[r], _ = oracle.decode_sequence(S[r], one, layer.variant)
            if r in sample:
                assert rel_err(o[r], o_ref[0]) <= tol, ("decode", r)
        np.copyto(n, (n + 1) % m)

    # a committed buffer of 0..3 tokens per request
    for _ in range(int(rng.integers(0, 4))):
        decode_round()
    for rnd in range(3):
        T = int(rng.integers(2, 9))
        parents = np.array([_random_tree(rng, T) for _ in range(B)], dtype=np.int32)
        if rnd == 0:
            parents[0] = np.arange(-1, T - 1)  # one chain among the trees
        tok = I.draw_tokens(rng, layer, (B, T))
        o = pool.verify_tree(req, parents, *token_tensors(tok, layer, slice(None))).cpu().numpy()
        for r in sample:
            o_ref = oracle.verify_tree(S[r], _row(tok, r), parents[r], layer.variant)
            assert rel_err(o[r], o_ref) <= tol, ("verify", rnd, r)
        accepted = rng.integers(-1, T, size=B)
        deepest = max(range(T), key=lambda j: (len(_path(parents[1], j)), j))
        accepted[1] = deepest  # a long path that is usually not the leading drafts
        pool.accept_tree(req, accepted)
        for r in range(B):
            S[r] = oracle.accept_tree(S[r], _row(tok, r), parents[r], int(accepted[r]),
                                      layer.variant)
            n[r] += len(_path(parents[r], int(accepted[r])))
            if n[r] >= m:
                n[r] = 0
        assert np.array_equal(pool.get_lengths(), n), rnd
        torch.cuda.synchronize()
        st = pool.state.cpu().numpy()
        for r in sample:
            if n[r] == 0:
                assert rel_err(st[r], S[r]) <= tol, ("state", rnd, r)
        for _ in range(2):
            decode_round()
        assert np.array_equal(pool.get_lengths(), n)
    pool.flush(req)
    torch.cuda.synchronize()
    st = pool.state.cpu().numpy()
    for r in sample:
        assert rel_err(st[r], S[r]) <= tol, ("final", r)
    assert np.array_equal(pool.get_device_lengths(), np.zeros(B))
    assert pool.get_error() is None


def test_tree_errors_and_chain_accept():
    kvb = kvb_mod()
    layer = I.Layer(I.GATED, 1, 1, 64, 64, "bf16")
    rng = np.random.default_rng(510)
    pool = make_pool(layer, 8, 2, 2, 8)
    for r in range(2):
        pool.set_request(r, r, [2 * r, 2 * r + 1])
    T = 3
    tok = I.draw_tokens(rng, layer, (2, T))
    args = token_tensors(tok, layer, slice(None))
    with pytest.raises(kvb.KvbError) as ex:  # a parent that is not an earlier draft
        pool.verify_tree([0, 1], [[-1, 0, 2], [-1, -1, -1]], *args)
    assert ex.value.status == kvb.KVB_E_ARG
    pool.verify_tree([0, 1], [[-1, 0, 0], [-1, -1, 1]], *args)
    with pytest.raises(kvb.KvbError) as ex:  # a tree needs kvb_accept_tree
        pool.accept([0, 1], [1, 1])
    assert ex.value.status == kvb.KVB_E_STATE
    with pytest.raises(kvb.KvbError) as ex:
        pool.accept_tree([0, 1], [0, 3])
    assert ex.value.status == kvb.KVB_E_ARG
    pool.accept_tree([0, 1], [2, 2])  # paths 0 -> 2 and 1 -> 2
    assert np.array_equal(pool.get_lengths(), [2, 2])
    # a chain verify accepted through kvb_accept_tree keeps drafts 0..j
    pool.verify([0, 1], *args)
    pool.accept_tree([0, 1], [1, -1])
    assert np.array_equal(pool.get_lengths(), [4, 2])
    assert pool.get_error() is None
