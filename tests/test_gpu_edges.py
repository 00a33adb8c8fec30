"""GPU edge cases: error statuses, degenerate calls, batch splitting, d=64 with grouped heads,
the device error word, and the copy probe."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import dev, make_pool, rel_err, token_tensors, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from kv_buffered_decoding_gb300 import kvb  # noqa: E402

SMALL_GDN = I.Layer(I.GATED_DELTA, 2, 4, 64, 64, "bf16", qk_dist="l2norm")


def _status(fn, *a, **k):
    try:
        fn(*a, **k)
    except kvb.KvbError as e:
        return e.status
    return kvb.KVB_OK


def test_error_statuses_and_empty_batch():
    layer = I.GATED_LAYER
    pool = make_pool(layer, 4, 4, 1, 4, num_slots=2)
    pool.state.zero_()
    pool.set_request(0, 0, [0])
    pool.set_request(1, -1, [1])
    rng = np.random.default_rng(0)
    tok = I.draw_tokens(rng, layer, (2,))
    a = token_tensors(tok, layer, slice(None))
    a1 = token_tensors(tok, layer, slice(0, 1))
    # empty batch: no launch, no error
    e = [t[:0] if t is not None else None for t in a]
    assert _status(pool.decode, [], *e) == kvb.KVB_OK
    # request kind checks
    assert _status(pool.decode, [1], *a1) == kvb.KVB_E_STATE
    assert _status(pool.short_ctx, [0], *a1) == kvb.KVB_E_STATE
    assert _status(pool.decode, [0, 0], *a) == kvb.KVB_E_ARG  # duplicate rows
    assert _status(pool.decode, [2], *a1) == kvb.KVB_E_STATE  # inactive
    assert _status(pool.decode, [9], *a1) == kvb.KVB_E_RANGE
    # ids at admission
    assert _status(pool.set_request, 2, 0, [2]) == kvb.KVB_E_RANGE   # slot owned by request 0
    assert _status(pool.set_request, 2, -1, [1]) == kvb.KVB_E_RANGE  # block owned by request 1
    assert _status(pool.set_request, 2, -1, [7]) == kvb.KVB_E_RANGE  # block out of range
    assert _status(pool.set_request, 0, -1, [2]) == kvb.KVB_E_STATE  # already active
    # capacity: the short request's buffer holds 4 tokens
    for _ in range(4):
        pool.short_ctx([1], *a1)
    assert _status(pool.short_ctx, [1], *a1) == kvb.KVB_E_CAPACITY
    assert pool.get_lengths()[1] == 4
    # verify bookkeeping: n + T must fit; a pending verify blocks decode; j <= T
    assert _status(pool.verify, [0], *[None if t is None else t[None, :1].expand(1, 5, *t.shape[1:])
                                       .contiguous() for t in a1]) == kvb.KVB_E_CAPACITY
    v1 = [None if t is None else t[None] for t in a1]
    pool.verify([0], *v1)
    assert _status(pool.decode, [0], *a1) == kvb.KVB_E_STATE
    assert _status(pool.accept, [0], [2]) == kvb.KVB_E_ARG
    assert _status(pool.accept, [1], [0]) == kvb.KVB_E_STATE  # nothing pending
    pool.accept([0], [1])
    assert pool.get_lengths()[0] == 1
    torch.cuda.synchronize()
    assert pool.get_error() is None
    assert np.array_equal(pool.get_device_lengths(), pool.get_lengths())


def test_batch_split_over_launch_rows():
    """600 rows exceed one launch's parameter block: the library splits the batch."""
    layer = I.Layer(I.GATED, 1, 1, 64, 64, "bf16")
    B, m = 600, 3
    rng = np.random.default_rng(1)
    pool = make_pool(layer, m, B, 1, 4)
    S0 = I.draw_state(rng, layer, B, scale=0.1)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, B - 1 - r, [r])  # reversed state slots
    tok = I.draw_tokens(rng, layer, (7, B))
    S_slot = S0[::-1].copy()  # request r's state lives in slot B-1-r
    o_ref, S_end, st = oracle.decode_sequence(S_slot, tok, layer.variant, keep_states=[5])
    outs = [pool.decode(np.arange(B), *token_tensors(tok, layer, t)).cpu().numpy() for t in range(7)]
    assert rel_err(np.stack(outs), o_ref) <= tol_for(layer)
    torch.cuda.synchronize()
    assert rel_err(pool.state.cpu().numpy()[::-1], st[5]) <= tol_for(layer)
    assert (pool.get_lengths() == 1).all()


def test_gdn_d64_grouped_heads_all_calls():
    """d=64, 2 q/k heads shared by 4 value heads: decode, verify/accept, flush, short ctx."""
    layer = SMALL_GDN
    m, bs, B = 5, 4, 6
    rng = np.random.default_rng(2)
    pool = make_pool(layer, m, B + 2, 4, bs, num_slots=B)
    S0 = I.draw_state(rng, layer, B)
    pool.state.copy_(torch.from_numpy(S0))
    perm = rng.permutation((B + 2) * 4)
    for r in range(B):
        pool.set_request(r, r, perm[4 * r:4 * r + 4])
    for r in (B, B + 1):
        pool.set_request(r, -1, perm[4 * r:4 * r + 4])
    req = np.arange(B)
    hist = {key: [] for key in ("q", "k", "v", "log_g", "beta")}
    outs, refs_idx = [], []
    tol = tol_for(layer)
    # 7 decode steps (one fold at step 5), then verify 3 drafts, accept ragged prefixes
    for t in range(7):
        tok = I.draw_tokens(rng, layer, (B,))
        outs.append(pool.decode(req, *token_tensors(tok, layer, slice(None))).cpu().numpy())
        for key in hist:
            hist[key].append(tok[key])
    H = {key: np.stack(v) for key, v in hist.items()}
    o_ref, S7, _ = oracle.decode_sequence(S0, H, layer.variant)
    assert rel_err(np.stack(outs), o_ref) <= tol
    drafts = I.draw_tokens(rng, layer, (B, 3))
    o = pool.verify(req, *[dev(drafts[k_], layer) for k_ in ("q", "k", "v")],
                    dev(drafts["log_g"], f32=True), dev(drafts["beta"], f32=True))
    dT = {key: np.swapaxes(val, 0, 1) for key, val in drafts.items()}
    o_ref = oracle.verify(S7, dT, layer.variant)
    assert rel_err(np.swapaxes(o.cpu().numpy(), 0, 1), o_ref) <= tol
    j = np.array([0, 1, 2, 3, 3, 2])
    pool.accept(req, j)
    S_acc = oracle.accept(S7, dT, j, layer.variant)
    # lengths: 7 tokens with m=5 -> 2 buffered, plus j; >= 5 folds
    expect = 2 + j
    expect[expect >= m] = 0
    assert np.array_equal(pool.get_lengths()[:B], expect)
    pool.flush(req)
    torch.cuda.synchronize()
    assert rel_err(pool.state.cpu().numpy(), S_acc) <= tol
    # short-context requests on the same layer
    sh = I.draw_tokens(rng, layer, (9, 2))
    so = [pool.short_ctx([B, B + 1], *token_tensors(sh, layer, t)).cpu().numpy() for t in range(9)]
    for i in range(2):
        ref = oracle.short_context({k_: v_[:, i] for k_, v_ in sh.items()}, layer.variant,
                                   layer.d_k, layer.d_v)
        assert rel_err(np.stack(so)[:, i], ref) <= tol
    assert pool.get_error() is None


def test_device_error_word_on_corrupt_table():
    """A block id corrupted in the device block table is caught by the kernel's own check:
    the CTA records (kind=1, request, value) and returns before using it; nothing faults.
    The first eight blocks of a request travel in the launch's row descriptors, so the
    corrupted entry is the ninth block (slots 16, 17 at 2 slots per block)."""
    layer = I.GATED_LAYER
    pool = make_pool(layer, 4, 2, 16, 2, num_slots=1)
    pool.set_request(0, -1, list(range(16)))
    pool.set_request(1, -1, list(range(16, 32)))
    rng = np.random.default_rng(3)
    tok = I.draw_tokens(rng, layer, (17, 2))
    outs = [pool.short_ctx([0, 1], *token_tensors(tok, layer, t)).cpu().numpy() for t in range(16)]
    torch.cuda.synchronize()
    # the block table is the first region of the metadata: request 0, block 8
    bad = torch.tensor([12345], dtype=torch.int32).view(torch.uint8).cuda()
    pool._meta_mem[32:36].copy_(bad)
    outs.append(pool.short_ctx([0, 1], *token_tensors(tok, layer, 16)).cpu().numpy())
    err = pool.get_error()
    assert err == (1, 0, 12345)
    assert pool.get_error() is None  # cleared
    # request 1 was served normally throughout
    ref = oracle.short_context({k_: (None if v_ is None else v_[:, 1]) for k_, v_ in tok.items()},
                               layer.variant, layer.d_k, layer.d_v)
    assert rel_err(np.stack(outs)[:, 1], ref) <= tol_for(layer)


def test_copy_probe():
    src = torch.randn(64 << 20, device="cuda")  # 256 MiB
    dst = torch.empty_like(src)
    kvb.copy_probe(src, dst)
    torch.cuda.synchronize()
    assert torch.equal(src, dst)
