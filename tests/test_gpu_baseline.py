"""GPU parity: the temporary-state verification baseline (recurrent pool, Figure 2).

Every draft's output, every temporary state (the state after drafts 0..j) and the
state after accepting a prefix are compared with the fp64 oracle; rows that accept
nothing keep their state bit for bit.
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


@pytest.mark.parametrize("layer", [
    I.Layer(I.GATED, 4, 4, 128, 128, "bf16"),
    I.Layer(I.GATED_DELTA, 2, 4, 128, 128, "bf16", qk_dist="l2norm"),
    I.Layer(I.GATED_DELTA, 1, 2, 64, 64, "f32", qk_dist="l2norm"),
], ids=["gated_d128", "gated_delta_d128", "gated_delta_d64_f32"])
def test_tempstate_verify_and_accept(layer):
    B, T = 6, 4
    rng = np.random.default_rng(70)
    S0 = I.draw_state(rng, layer, B)
    pool = make_pool(layer, 0, B, 1, 8)
    pool.state.copy_(torch.from_numpy(S0))
    for r in range(B):
        pool.set_request(r, B - 1 - r, [])
    S_slot = S0[::-1].copy()  # request r lives in slot B-1-r
    req = np.arange(B)
    S_hist = S_slot.astype(np.float64)
    tol = tol_for(layer)
    for rnd in range(5):
        tok = I.draw_tokens(rng, layer, (B, T))
        o, temp = pool.verify_tempstate(req, dev(tok["q"], layer), dev(tok["k"], layer),
                                        dev(tok["v"], layer), dev(tok["log_g"], f32=True),
                                        dev(tok["beta"], f32=True))
        drafts = {key: (None if val is None else np.swapaxes(val, 0, 1)) for key, val in tok.items()}
        o_ref, _, states = oracle.decode_sequence(S_hist, drafts, layer.variant,
                                                  keep_states=range(T))
        assert rel_err(np.swapaxes(o.cpu().numpy(), 0, 1), o_ref) <= tol
        tp = temp.cpu().numpy()
        for j in range(T):
            assert rel_err(tp[:, j], states[j]) <= tol, (rnd, j)
        before = pool.state.clone()
        j = rng.integers(0, T + 1, size=B)
        j[0] = 0
        pool.accept_tempstate(req, j, temp)
        torch.cuda.synchronize()
        S_hist = oracle.accept(S_hist, drafts, j, layer.variant)
        got = pool.state.cpu().numpy()[::-1]
        assert rel_err(got, S_hist) <= tol
        # request 0 accepted nothing: its slot (B-1) is untouched
        assert torch.equal(pool.state[B - 1], before[B - 1])
    assert pool.get_error() is None
