"""GPU: the allocation-free temporary-state verify (kvb_verify_tempstate_static)
against the allocating one (kvb_verify_tempstate + kvb_accept_tempstate).

Two pools start from the same states.  One takes the allocating path with a
caller-owned temporary-state tensor; the other calls the allocation-free entry
point through the C ABI, whose temporary states live in the library's fixed
device array.  Two calls in a row are compared (the second over a different
batch, so it runs over what the first left in the array): draft outputs and the
states after accepting a prefix must agree within the test tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest

from kv_buffered_decoding_gb300 import inputs as I
from tests.gpu_harness import dev, kvb_mod, make_pool, rel_err, tol_for

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)


def _pools(layer, R, S0):
    pools = []
    for _ in range(2):
        pool = make_pool(layer, 0, R, 1, 8)
        pool.state.copy_(torch.from_numpy(S0))
        for r in range(R):
            pool.set_request(r, R - 1 - r, [])
        pools.append(pool)
    return pools


@pytest.mark.parametrize("layer", [
    I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm"),
    I.Layer(I.GATED, 1, 2, 64, 64, "f32"),
], ids=["gated_delta_d128_bf16", "gated_d64_f32"])
def test_static_matches_allocating_path(layer):
    R = 8
    rng = np.random.default_rng(91)
    S0 = I.draw_state(rng, layer, R)
    ref, nal = _pools(layer, R, S0)
    tol = tol_for(layer)
    for call, (rows, T) in enumerate([(np.arange(R), 4), (np.array([6, 1, 3]), 3)]):
        tok = I.draw_tokens(rng, layer, (len(rows), T))
        args = (dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
                dev(tok["log_g"], f32=True), dev(tok["beta"], f32=True))
        j = rng.integers(0, T + 1, size=len(rows))
        j[0] = 0
        o_ref, temp = ref.verify_tempstate(rows, *args)
        ref.accept_tempstate(rows, j, temp)
        before = nal.state.clone()
        o = nal.verify_tempstate_static(rows, *args, n_accepted=j)
        torch.cuda.synchronize()
        assert rel_err(o.cpu().numpy(), o_ref.cpu().numpy()) <= tol, call
        assert rel_err(nal.state.cpu().numpy(), ref.state.cpu().numpy()) <= tol, call
        slot0 = R - 1 - int(rows[0])  # the first row accepted nothing
        assert torch.equal(nal.state[slot0], before[slot0]), call
    # without n_accepted the call only verifies: the states stay as they are
    rows = np.arange(R)
    tok = I.draw_tokens(rng, layer, (R, 2))
    args = (dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
            dev(tok["log_g"], f32=True), dev(tok["beta"], f32=True))
    o_ref, _ = ref.verify_tempstate(rows, *args)
    before = nal.state.clone()
    o = nal.verify_tempstate_static(rows, *args)
    torch.cuda.synchronize()
    assert rel_err(o.cpu().numpy(), o_ref.cpu().numpy()) <= tol
    assert torch.equal(nal.state, before)
    assert nal.get_error() is None and ref.get_error() is None


def test_static_rejects_oversized_batch():
    kvb = kvb_mod()
    layer = I.Layer(I.GATED, 2, 4, 128, 128, "bf16")
    per_row_draft = layer.n_v_heads * layer.d_k * layer.d_v * 4
    T = 4
    B = kvb.KVB_STATIC_TEMP_BYTES // (per_row_draft * T) + 1
    rng = np.random.default_rng(92)
    pool = make_pool(layer, 0, B, 1, 8)
    for r in range(B):
        pool.set_request(r, r, [])
    before = pool.state.clone()
    tok = I.draw_tokens(rng, layer, (B, T))
    args = (dev(tok["q"], layer), dev(tok["k"], layer), dev(tok["v"], layer),
            dev(tok["log_g"], f32=True), dev(tok["beta"], f32=True))
    with pytest.raises(kvb.KvbError) as ex:
        pool.verify_tempstate_static(np.arange(B), *args, n_accepted=np.full(B, T))
    assert ex.value.status == kvb.KVB_E_CAPACITY
    torch.cuda.synchronize()
    assert torch.equal(pool.state, before)
