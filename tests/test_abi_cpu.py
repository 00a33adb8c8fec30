"""CPU-only checks of the boundary: the library loads, exports every symbol the header
declares, and rejects bad arguments on the host before touching a GPU.  Plus the
benchmark's byte arithmetic and its multi-rank timing logic (gloo, 2 ranks)."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvb():
    from kv_buffered_decoding_gb300 import build, kvb as mod
    build.build()
    mod.load_library()
    return mod


def _declared():
    with open(os.path.join(ROOT, "include", "kvb.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvb_[a-z_]+)\s*\(", text)))


def test_header_symbols_exported(kvb):
    declared = _declared()
    assert len(declared) >= 16
    lib = ctypes.CDLL(kvb.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), name
    assert sorted(kvb.EXPORTS) == declared


def test_version_and_strerror(kvb):
    assert "sm_103a" in kvb.kvb_version()
    for st in (0, -1, -2, -3, -4, -5, -6, -7):
        assert kvb.kvb_strerror(st) != "unknown status"
    assert kvb.kvb_strerror(-99) == "unknown status"


def test_layout_arithmetic(kvb):
    cfg = kvb.make_config(kvb.KVB_GATED_DELTA, kvb.KVB_BF16, 16, 32, 128, 128, 8, 8, 256, 256, 256, 1)
    lay = kvb.kvb_pool_layout(cfg)
    assert lay.state_bytes == 256 * 32 * 128 * 128 * 4  # 512 MiB
    assert lay.state_slot_stride == 32 * 128 * 128 * 4
    rows = 256 * 8
    assert lay.v_off >= lay.k_off + rows * 16 * 128 * 2
    assert lay.u_off >= lay.v_off + rows * 32 * 128 * 2
    assert lay.logg_off >= lay.u_off + rows * 32 * 128 * 4
    assert lay.kv_bytes >= lay.beta_off + rows * 32 * 4
    for off in (lay.k_off, lay.v_off, lay.u_off, lay.logg_off, lay.beta_off, lay.kv_bytes):
        assert off % 256 == 0
    # no pseudo-value region for the gated variant
    cfg.variant = kvb.KVB_GATED
    lay2 = kvb.kvb_pool_layout(cfg)
    assert lay2.logg_off == lay2.u_off


@pytest.mark.parametrize("field,value,status", [
    ("variant", 3, -1), ("kv_dtype", 2, -1), ("n_v_heads", 24, -1), ("d_k", 96, -7),
    ("d_v", 64, -7), ("m", -1, -1), ("m", 65, -1), ("block_size", 0, -1), ("max_requests", 0, -1),
])
def test_layout_rejects_bad_config(kvb, field, value, status):
    cfg = kvb.make_config(kvb.KVB_GATED_DELTA, kvb.KVB_BF16, 16, 32, 128, 128, 8, 8, 16, 4, 4, 1)
    setattr(cfg, field, value)
    with pytest.raises(kvb.KvbError) as e:
        kvb.kvb_pool_layout(cfg)
    assert e.value.status == status


def test_host_side_argument_errors(kvb):
    lib = kvb.load_library()
    cfg = kvb.make_config(kvb.KVB_GATED, kvb.KVB_BF16, 16, 16, 128, 128, 8, 8, 16, 4, 4, 1)
    h = ctypes.c_void_p()
    # missing or misaligned metadata region: rejected before any CUDA call
    assert lib.kvb_alloc_pool(ctypes.byref(cfg), 256, 256, None, ctypes.byref(h)) == -1
    assert lib.kvb_alloc_pool(ctypes.byref(cfg), 256, 256, 257, ctypes.byref(h)) == -1
    assert lib.kvb_alloc_pool(ctypes.byref(cfg), 256, 256, 256, None) == -1
    assert not h.value
    ids = (ctypes.c_int32 * 1)(0)
    assert lib.kvb_decode(None, 1, ids, 16, 16, 16, 16, None, 16, 1, None) == -1
    assert lib.kvb_flush(None, 1, ids, None) == -1
    assert lib.kvb_accept(None, 1, ids, ids, None) == -1
    assert lib.kvb_get_lengths(None, ids) == -1
    assert lib.kvb_copy_probe(16, 32, 15, None) == -1   # size not a multiple of 16
    assert lib.kvb_copy_probe(16, 40, 32, None) == -1   # misaligned destination
    assert lib.kvb_copy_probe(16, 32, 0, None) == 0     # nothing to copy


def test_step_bytes_cycle_average():
    """Staggered occupancy: every step moves the cycle-average bytes (2,448,768 B per
    request-step at the B=256, Hk=16, Hv=32, d=128, m=8 shape)."""
    import bench
    w = bench.WORKLOAD
    lengths = np.arange(w.batch) % w.m
    assert bench.step_bytes(w, lengths) == 2_448_768 * w.batch
    # cycle-aligned start: 8 steps sum to the same total
    n = np.zeros(w.batch, dtype=np.int64)
    total = 0
    for _ in range(w.m):
        total += bench.step_bytes(w, n)
        n = (n + 1) % w.m
    assert total == 2_448_768 * w.batch * w.m


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [10.0, 25.0][rank]
    worst = bench.max_over_ranks(ms, dist)
    rate = bench.job_rate(world, 256, 100, worst)
    out.put((rank, worst, rate))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_timing_gloo():
    import multiprocessing as mp
    import socket
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, worst, rate in res:
        assert worst == 25.0
        assert rate == pytest.approx(2 * 256 * 100 / 0.025)


def test_prefill_wait_limit_hook(kvb):
    lib = kvb.load_library()
    assert lib.kvb_set_prefill_wait_limit(-1) == kvb.KVB_E_ARG
    assert lib.kvb_set_prefill_wait_limit(5) == kvb.KVB_OK
    assert lib.kvb_set_prefill_wait_limit(0) == kvb.KVB_OK
