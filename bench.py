"""Benchmark: buffered gated-delta decode, tokens/s per layer, and achieved HBM bandwidth.

Workload: gated delta rule layer with 16 q/k heads shared by 32 value heads,
d_k = d_v = 128, bf16 q/k/v and buffer, fp32 state, B = 256 requests, buffer
size m = 8.  A step is one decode step of all B requests (one kvb_decode
launch), with the fold of the requests whose buffer fills in that step.
Request r starts at buffer occupancy r mod m, so every step holds B/m requests
at each occupancy 0..m-1 and B/m folds: each step costs the cycle average.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Under torchrun (N > 1) every rank runs its
own B requests on its own GPU (weak scaling, no data-path collective); the
reported time is the maximum over ranks.
"""
from __future__ import annotations

import os

for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import statistics  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_buffered_decoding_gb300 import inputs as I  # noqa: E402

WORKLOAD = I.WORKLOADS["gdn_B256_Hk16_Hv32_d128"]
METRIC = "decode tok/s per layer (B=256, m=8) and achieved HBM GB/s vs peak"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
TF32_PER_BF16 = 1.1 / 2.25  # nominal dense tf32 / bf16 tensor rates of the part
N_BANK = 8  # distinct input token sets cycled through the timed steps


def workload_config(w=WORKLOAD):
    L = w.layer
    return {"workload": f"gated_delta_decode_B{w.batch}_Hk{L.n_qk_heads}_Hv{L.n_v_heads}"
                        f"_d{L.d_k}_m{w.m}_bf16",
            "batch": w.batch, "n_qk_heads": L.n_qk_heads, "n_v_heads": L.n_v_heads,
            "d_k": L.d_k, "d_v": L.d_v, "m": w.m, "variant": "gated_delta",
            "kv_dtype": "bf16", "state_dtype": "f32", "occupancy": "staggered (r mod m)",
            "l2": "inputs larger than L2: 512 MiB of state read per step, no flush needed"}


def step_bytes(w, lengths):
    """Algorithmic HBM bytes of one decode step given each request's occupancy before it.

    Per request: state read, q, the new token (k, v, log-gate, beta) read and
    appended, the n buffered tokens (raw k, v, gate, beta) read, o written, and
    the state written back when the step folds.
    """
    L = w.layer
    S = L.n_v_heads * L.d_k * L.d_v * 4
    entry = L.n_qk_heads * L.d_k * 2 + L.n_v_heads * L.d_v * 2 + 2 * L.n_v_heads * 4
    q = L.n_qk_heads * L.d_k * 2
    o = L.n_v_heads * L.d_v * 4
    n = np.asarray(lengths, dtype=np.int64)
    folds = int(np.count_nonzero(n + 1 >= w.m))
    return int(len(n) * (S + q + 2 * entry + o) + int(n.sum()) * entry + folds * S)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for key in ("hbm_gbs", "hbm_GBps", "hbm"):
                if key in d and isinstance(d[key], (int, float)):
                    return float(d[key]), "of measured (MEASURED_PEAKS.json hbm_gbs)"
        except (OSError, ValueError):
            pass
    return FALLBACK_HBM_GBS, "of fallback (6.8 TB/s, no MEASURED_PEAKS.json)"


def tensor_peak_bf16():
    """Dense bf16 tensor peak (TFLOP/s): the measured cuBLAS burst rate, else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for key in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
                if key in d and isinstance(d[key], (int, float)):
                    return float(d[key]), "of measured (MEASURED_PEAKS.json bf16_tflops)"
        except (OSError, ValueError):
            pass
    return FALLBACK_BF16_TFLOPS, "of fallback (1.9 PFLOP/s bf16)"


def tensor_peak_tf32():
    """Dense tf32 tensor peak (TFLOP/s): the measured bf16 GEMM burst rate times the
    nominal tf32/bf16 ratio, or the fallback bf16 figure times the same ratio."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for key in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
                if key in d and isinstance(d[key], (int, float)):
                    return float(d[key]) * TF32_PER_BF16, \
                        "of measured bf16 burst x nominal tf32/bf16 ratio"
        except (OSError, ValueError):
            pass
    return FALLBACK_BF16_TFLOPS * TF32_PER_BF16, \
        "of fallback (1.9 PFLOP/s bf16 x nominal tf32/bf16 ratio)"


def prefill_flops(L, n_tokens, chunk=64):
    """Arithmetic of the chunked form per call: per chunk and value head, Y = [Q; K] S
    (K rows for the delta rule only), the masked Gram triangles, the forward
    substitution (delta rule), the intra-chunk output and the state update; two flops
    per multiply-add.  n_tokens counts the prompt tokens of all requests."""
    C, dk, dv = chunk, L.d_k, L.d_v
    delta = L.variant == I.GATED_DELTA
    tri_incl, tri_strict = C * (C + 1) // 2, C * (C - 1) // 2
    per_chunk = (2 * (2 if delta else 1) * C * dk * dv      # Y
                 + 2 * tri_incl * dk                         # Mq
                 + (2 * tri_strict * dk if delta else 0)     # Mk
                 + (2 * tri_strict * dv if delta else 0)     # substitution
                 + 2 * tri_incl * dv                         # O intra-chunk
                 + 2 * C * dk * dv)                          # state update
    return per_chunk * (n_tokens / C) * L.n_v_heads


def kernel_hash():
    h = hashlib.sha256()
    for rel in ("kv_buffered_decoding_gb300/csrc/decode_stream.cu",
                "kv_buffered_decoding_gb300/csrc/kvb_device.cuh"):
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic():
    """DRAM bytes per launch of the decode kernel from the committed ncu summary, if it
    was taken on the current kernel source; else None."""
    path = os.path.join(ROOT, "profiles", "decode_gdn_B256_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_hash") != kernel_hash():
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open("/tmp/kvb_clocks_%d.csv" % os.getpid(), "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.out:
            self.out.close()

    def summary(self):
        if self.proc is None or self.out is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.out.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for name, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(name)
        os.unlink(self.out.name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "power_w_median": statistics.median(power), "samples": len(sm),
                "reasons": sorted(reasons)}


def max_over_ranks(ms, dist=None):
    """The slowest rank's time: every rank ran its own requests, so the job ends with it."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(ms)
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(world, batch, steps, elapsed_ms):
    """Whole-job tokens/s: every rank decodes `batch` requests for `steps` steps."""
    return world * batch * steps / (elapsed_ms / 1e3)


# --------------------------------------------------------------------------- CPU arm
def oracle_rate(w, budget_s, reqs_per_step=8, seed=11, max_steps=None):
    """The fp64 oracle (as it stands) on a bounded sample of the workload: consecutive
    decode steps of `reqs_per_step` requests (all 32 heads).  Returns (tok/s, steps, secs)."""
    import oracle
    rng = np.random.default_rng(seed)
    L = w.layer
    S = I.draw_state(rng, L, reqs_per_step).astype(np.float64)
    steps, t0 = 0, time.perf_counter()
    while True:
        tok = I.draw_tokens(rng, L, (1, reqs_per_step))
        _, S, _ = oracle.decode_sequence(S, tok, L.variant)
        steps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and steps >= max_steps):
            break
    return reqs_per_step * steps / el, steps, el


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _oracle_worker(job):
    """One host process of the all-core oracle run: its own requests (seed), timed alone."""
    budget_s, reqs, max_steps, seed = job
    rate, steps, el = oracle_rate(WORKLOAD, budget_s, reqs_per_step=reqs, seed=seed,
                                  max_steps=max_steps)
    return reqs * steps, el


def oracle_rate_all_cores(budget_s, reqs_per_step=8, max_steps=None, cores=None):
    """The oracle (as it stands, one thread per process) on every host core at once:
    one spawned process per core, each decoding its own disjoint requests for the same
    budget.  Returns (aggregate tok/s, cores, tokens, slowest process's seconds)."""
    import multiprocessing as mp
    from concurrent.futures import ProcessPoolExecutor
    cores = cores or host_cores()
    jobs = [(budget_s, reqs_per_step, max_steps, 100 + i) for i in range(cores)]
    # spawn, not fork: this process has initialised CUDA; a worker that dies raises
    # BrokenProcessPool here instead of being restarted
    with ProcessPoolExecutor(cores, mp_context=mp.get_context("spawn")) as ex:
        res = list(ex.map(_oracle_worker, jobs))
    tokens = sum(t for t, _ in res)
    slowest = max(el for _, el in res)
    return tokens / slowest, cores, tokens, slowest


def run_reference(args, rank, world):
    """The oracle as the reference arm, on every host core, in this workload's unit.

    A step is one decode token for a few requests in each of C processes (one per host
    core, disjoint requests); the value is all processes' tokens over the slowest
    process's time.  The one-core rate is reported beside it."""
    if rank != 0:
        return
    w = WORKLOAD
    for _ in range(max(args.warmup, 0)):
        oracle_rate(w, float("inf"), reqs_per_step=1, max_steps=1)
    # size each step so the K timed steps take about a minute
    probe, _, _ = oracle_rate(w, float("inf"), reqs_per_step=1, max_steps=1)
    per_req = 1.0 / probe
    reqs = int(max(1, min(8, round(60.0 / max(args.steps, 1) / per_req))))
    value, cores, tokens, el = oracle_rate_all_cores(float("inf"), reqs_per_step=reqs,
                                                     max_steps=args.steps)
    steps = args.steps
    one, one_steps, one_el = oracle_rate(w, 10.0, reqs_per_step=reqs)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tok/s",
            "n_gpus": world, "steps": steps, "warmup": args.warmup,
            "ms_per_step": 1e3 * el / steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(),
            "cpu_baseline": {"value": value, "unit": "tok/s", "cores": cores, "kind": "oracle",
                             "sample": f"{cores} processes (one per host core), each {reqs} "
                                       f"request(s) x 32 heads per step, {steps} steps, fp64 "
                                       "per-token recurrence (numpy, one thread each)",
                             "one_core": {"value": one, "cores": 1,
                                          "sample": f"{reqs} request(s) x 32 heads, {one_steps} "
                                                    f"steps ({one_el:.1f} s), one process"}},
            "e2e": {"value": value, "unit": "tok/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- other rows
def _entry_bytes(L, esz=2):
    return L.n_qk_heads * L.d_k * esz + L.n_v_heads * L.d_v * esz + 2 * L.n_v_heads * 4


def measure_paths(kvb, torch, dev, peak):
    """Time the other calls of the path on this GPU against the same HBM roofline.

    verify: T = 4 drafts per request against the stored state, accepted with j = 0 so
    every round sees the same buffer; flush: fold 8 buffered tokens per request into the
    state; short_ctx: buffer-only decode of requests holding 32..44 tokens.  Each entry
    reports microseconds per call, algorithmic GB/s (raw q/k/v/gate/beta/state/output
    bytes, as for decode) and the fraction of the peak.
    """
    out = {}
    stream = torch.cuda.current_stream(dev)
    # figures whose data fits in L2 are labelled L2-assisted; the size they fit in
    out["l2_cache_bytes"] = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0))

    def checked_close(p):
        """Release a pool after reading its device error word: a timing taken while
        a kernel reported an error is not a result."""
        err = p.get_error()
        p.close()
        if err is not None:
            raise RuntimeError(f"device error during the path timings: {err}")

    def timed(fn, reps):
        """GPU time per call of `reps` back-to-back calls.  A sleep kernel holds the
        stream while the host enqueues them, so the host's per-call work (argument
        checks, row descriptors, launches) stays outside the events."""
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(20_000_000)  # about 10 ms: far longer than enqueueing the calls
        a.record(stream)
        for _ in range(reps):
            fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / reps * 1e3

    l2_flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2_clean = torch.ones(64 << 20, dtype=torch.int32, device=dev)

    def timed_cold(fn, reps):
        """Median GPU time of single calls, each after an L2 flush and a sleep kernel
        that keeps the host's launch latency out of the events.  The flush writes
        256 MiB, then reads another 256 MiB, so the write-backs of its dirty lines
        happen before the timed call and not inside it."""
        times = []
        for _ in range(reps):
            l2_flush.fill_(1)
            l2_clean.max()
            torch.cuda._sleep(2_000_000)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
        return statistics.median(times)

    def tokens(L, lead, seed):
        t = I.draw_tokens(np.random.default_rng(seed), L, lead)
        res = [torch.from_numpy(t[k_]).to(torch.bfloat16).to(dev) for k_ in ("q", "k", "v")]
        res.append(None if t["log_g"] is None else torch.from_numpy(t["log_g"]).to(dev))
        res.append(None if t["beta"] is None else torch.from_numpy(t["beta"]).to(dev))
        return res

    def pool_for(L, B, m, nb, bs=8, slots=True):
        v = kvb.KVB_GATED_DELTA if L.variant == I.GATED_DELTA else kvb.KVB_GATED
        cfg = kvb.make_config(v, kvb.KVB_BF16, L.n_qk_heads, L.n_v_heads, L.d_k, L.d_v, m, bs,
                              B * nb, B if slots else 0, B, nb)
        pool = kvb.Pool(cfg, device=dev)
        if slots:
            pool.state.normal_(0.0, 1.0 / np.sqrt(L.d_k))
        for r in range(B):
            blocks = list(range(r * nb, (r + 1) * nb)) if m > 0 or not slots else []
            pool.set_request(r, r if slots else -1, blocks)
        return pool

    def rec(name, us, nbytes, note):
        gbs = nbytes / us / 1e3
        out[name] = {"us_per_call": us, "gbs": gbs, "frac": gbs / peak, "bytes": nbytes,
                     "note": note}

    # verify: gated delta bench layer at B=256 (HBM-bound) and the gated layer at B=64
    for L, B, tag in ((I.GDN_LAYER, 256, "verify_gated_delta_B256_T4"),
                      (I.GATED_LAYER, 64, "verify_gated_B64_T4")):
        T, m, n0 = 4, 8, 3
        pool = pool_for(L, B, m, 2)
        req = np.arange(B, dtype=np.int32)
        pre = tokens(L, (B,), 5)
        for _ in range(n0):
            pool.decode(req, *pre)
        drafts = tokens(L, (B, T), 6)
        zero = np.zeros(B, dtype=np.int32)

        def one():
            pool.verify(req, *drafts)
            pool.accept(req, zero)
        us = timed(one, 50)
        S = L.n_v_heads * L.d_k * L.d_v * 4
        q = L.n_qk_heads * L.d_k * 2
        o = L.n_v_heads * L.d_v * 4
        e = _entry_bytes(L)
        nbytes = B * (S + T * (q + 2 * e + o) + n0 * e)
        rec(tag, us, nbytes, "verify + accept(0) per round; state %d MiB%s" % (
            B * S >> 20, " (L2-resident: L2-assisted)" if B * S < 100 * 2 ** 20 else ""))
        checked_close(pool)

    # draft tree: 8 drafts as a binary tree of depth 4 (every request the same shape)
    # against a chain of 8, gated delta layer at B=256; accept(-1 / 0) keeps the buffer
    L, B, T, n0 = I.GDN_LAYER, 256, 8, 3
    pool = pool_for(L, B, 8, 2)
    req = np.arange(B, dtype=np.int32)
    pre = tokens(L, (B,), 5)
    for _ in range(n0):
        pool.decode(req, *pre)
    drafts = tokens(L, (B, T), 7)
    parents = np.tile(np.array([-1, 0, 0, 1, 1, 2, 2, 3], dtype=np.int32), (B, 1))
    none = np.full(B, -1, dtype=np.int32)
    zero = np.zeros(B, dtype=np.int32)
    o_t = torch.empty(B, T, L.n_v_heads, L.d_v, dtype=torch.float32, device=dev)

    def tree_round():
        pool.verify_tree(req, parents, *drafts, o=o_t)
        pool.accept_tree(req, none)

    def chain_round():
        pool.verify(req, *drafts, o=o_t)
        pool.accept(req, zero)
    us_tree = timed(tree_round, 30)
    us_chain = timed(chain_round, 30)
    S = L.n_v_heads * L.d_k * L.d_v * 4
    q = L.n_qk_heads * L.d_k * 2
    o = L.n_v_heads * L.d_v * 4
    e = _entry_bytes(L)
    nbytes = B * (S + T * (q + 2 * e + o) + n0 * e)
    rec("verify_tree_gated_delta_B256_T8", us_tree, nbytes,
        "binary draft tree of depth 4 (8 drafts) + accept_tree(-1) per round; one launch "
        "of 256 rows")
    out["verify_tree_gated_delta_B256_T8"]["chain_T8_us"] = us_chain
    del o_t
    checked_close(pool)

    # verify latency against the number of drafts: buffered verify vs the recurrent
    # temporary-state baseline (Figure 2), gated delta layer at B=256, plus the memory
    # each needs per request (state + buffer slots vs state + T temporary states)
    L, B = I.GDN_LAYER, 256
    S = L.n_v_heads * L.d_k * L.d_v * 4
    slot_bytes = _entry_bytes(L) + L.n_v_heads * L.d_v * 4  # raw k/v/gate/beta + pseudo-value
    cmp = {}
    for T in (2, 4, 6, 8):
        pool = pool_for(L, B, 8, 2)
        base = pool_for(L, B, 0, 1)
        base.state.copy_(pool.state)
        req = np.arange(B, dtype=np.int32)
        pre = tokens(L, (B,), 9)
        for _ in range(3):
            pool.decode(req, *pre)
        drafts = tokens(L, (B, T), 10 + T)
        zero = np.zeros(B, dtype=np.int32)
        temp = torch.empty(B, T, L.n_v_heads, L.d_k, L.d_v, dtype=torch.float32, device=dev)
        o = torch.empty(B, T, L.n_v_heads, L.d_v, dtype=torch.float32, device=dev)

        def kvb_round():
            pool.verify(req, *drafts, o=o)
            pool.accept(req, zero)

        us_kvb = timed(kvb_round, 30)
        us_base = timed(lambda: base.verify_tempstate(req, *drafts, temp=temp, o=o), 30)
        cmp[str(T)] = {"buffered_us": us_kvb, "tempstate_us": us_base,
                       "buffered_bytes_per_request": S + (8 - 1 + T) * slot_bytes,
                       "tempstate_bytes_per_request": (1 + T) * S}
        del temp
        checked_close(pool)
        checked_close(base)
    out["verify_vs_tempstate_gated_delta_B256"] = cmp

    # Figure 3 of the page: decode latency averaged over a full buffer cycle
    # (occupancies 0..m-1 and the fold) for each buffer size m, normalised to m = 0
    # (recurrent decoding); scalar-gated layer, 16 heads, d = 128, B = 256 and the
    # 32-request batch of the sweep workload (whose 32 MiB of state stays in L2)
    for B in (256, 32):
        L = I.GATED_LAYER
        sweep = {}
        for m in (0, 2, 4, 8, 16):
            nbpr = max(1, -(-m // 8))
            pool = pool_for(L, B, m, nbpr)
            req = np.arange(B, dtype=np.int32)
            toks = tokens(L, (B,), 20 + m)
            cycle = max(m, 1)
            us = timed(lambda: pool.decode(req, *toks), 8 * cycle)
            sweep[str(m)] = us
            checked_close(pool)
        out["fig3_gated_B%d" % B] = {
            "us_per_step": sweep,
            "normalised_to_m0": {m_: v / sweep["0"] for m_, v in sweep.items()},
            "note": "timed over whole cycles from a cycle-aligned start (every request folds "
                    "on the same step); state %d MiB%s" % (
                        B * L.n_v_heads * L.d_k * L.d_v * 4 >> 20,
                        " (L2-assisted)" if B * L.n_v_heads * L.d_k * L.d_v * 4 < 100 * 2 ** 20 else "")}

    # flush: 8 buffered tokens per request folded into the state (gated delta, B=256)
    L, B = I.GDN_LAYER, 256
    pool = pool_for(L, B, 8, 1)
    req = np.arange(B, dtype=np.int32)
    toks = tokens(L, (B,), 7)
    S = L.n_v_heads * L.d_k * L.d_v * 4
    e = _entry_bytes(L)
    times = []
    for rep in range(8):
        for _ in range(8):
            pool.decode(req, *toks, auto_flush=False)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            torch.cuda._sleep(2_000_000)  # keeps the host's launch latency out of the events
        a.record(stream)
        pool.flush(req)
        b.record(stream)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b) * 1e3)
    us = statistics.median(times[2:])
    rec("flush_gated_delta_B256_L8", us, B * (2 * S + 8 * e), "one kvb_flush of 8 tokens per request")
    checked_close(pool)

    # short context: buffer-only decode, gated layer, B=256 requests holding 32..44 tokens
    L, B = I.GATED_LAYER, 256
    pool = pool_for(L, B, 8, 8, slots=False)
    req = np.arange(B, dtype=np.int32)
    toks = tokens(L, (B,), 8)
    for _ in range(32):
        pool.short_ctx(req, *toks)
    base = pool.get_lengths()[:B].astype(np.int64)
    reps = 13  # lengths go from base to base + 12, each call after an L2 flush
    us_single = timed_cold(lambda: pool.short_ctx(req, *toks), reps)
    checked_close(pool)

    def flushed_sequence(fn=None):
        """GPU time of `reps` L2 flushes, each followed by one call of fn if given,
        queued back to back as a stream of work would be."""
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(2_000_000)
        a.record(stream)
        for _ in range(reps):
            l2_flush.fill_(1)
            l2_clean.max()
            if fn is not None:
                fn()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b) * 1e3

    # the same calls queued back to back (each after the flush): the difference to
    # the flushes alone, per call; fresh pools so that each sequence covers 32..44
    # tokens again; median of five
    piped = []
    for _ in range(5):
        p2 = pool_for(L, B, 8, 8, slots=False)
        for _ in range(32):
            p2.short_ctx(req, *toks)
        with_calls = flushed_sequence(lambda: p2.short_ctx(req, *toks))
        alone = flushed_sequence()
        piped.append((with_calls - alone) / reps)
        checked_close(p2)
    us = statistics.median(piped)
    mean_n = float(base.mean()) + (reps - 1) / 2.0
    q = L.n_qk_heads * L.d_k * 2
    o = L.n_v_heads * L.d_v * 4
    e = _entry_bytes(L)
    rec("short_ctx_gated_B256_n32to44", us, int(B * (q + 2 * e + o + mean_n * e)),
        "buffer-only decode, no state; buffer reads dominate; cold L2: each call after an "
        "L2 flush, calls and flushes queued back to back, the flushes' own time subtracted "
        "(median of five sequences of 13)")
    out["short_ctx_gated_B256_n32to44"]["us_single_call"] = us_single
    out["short_ctx_gated_B256_n32to44"]["single_call_note"] = (
        "one call between two events after a sleep kernel: adds the event and launch floor, "
        "about 4-6 us for an empty kernel on this GPU")

    # Figure 5 of the pages: per-step latency against context length for KV-only
    # decoding (short context: the buffer alone, no state), recurrent decoding
    # (m = 0) and buffered decoding (m = 8, averaged over a whole cycle), gated layer,
    # B = 256.  Every step runs on a cold L2, as one layer's step among a model's
    # layers would: k steps, each after an L2 flush, queued back to back, minus the
    # flushes alone.  KV-only contexts stop at 60..63 tokens (64-slot buffers); a
    # request that outgrows them is promoted to a state (kvb_promote).
    def cold_per_call(fn, k):
        def seq(f):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda._sleep(2_000_000)
            a.record(stream)
            for _ in range(k):
                l2_flush.fill_(1)
                l2_clean.max()
                if f is not None:
                    f()
            b.record(stream)
            torch.cuda.synchronize()
            return a.elapsed_time(b) * 1e3
        return (seq(fn) - seq(None)) / k

    L, B = I.GATED_LAYER, 256
    req = np.arange(B, dtype=np.int32)
    toks = tokens(L, (B,), 30)
    kv_only = {}
    for ctx in (16, 32, 48, 60):
        vals = []
        for _ in range(3):
            pk = pool_for(L, B, 8, 8, slots=False)
            for _ in range(ctx - 1):
                pk.short_ctx(req, *toks)
            vals.append(cold_per_call(lambda: pk.short_ctx(req, *toks), 4))  # contexts ctx .. ctx + 3
            checked_close(pk)
        kv_only[str(ctx)] = statistics.median(vals)
    by_m = {}
    for m_ in (0, 8):
        vals = []
        for _ in range(3):
            pm = pool_for(L, B, m_, 1)
            k_ = max(m_, 4)  # a whole cycle of occupancies 0..m-1 (the last step folds)
            vals.append(cold_per_call(lambda: pm.decode(req, *toks), k_))
            checked_close(pm)
        by_m[m_] = statistics.median(vals)
    out["fig5_context_gated_B256"] = {
        "kv_only_us": kv_only, "recurrent_m0_us": by_m[0], "buffered_m8_us": by_m[8],
        "kv_only_normalised_to_m0": {c: v / by_m[0] for c, v in kv_only.items()},
        "buffered_m8_normalised_to_m0": by_m[8] / by_m[0],
        "note": "per-step GPU time, each step after an L2 flush (flush time subtracted); KV-only at "
                "context c averages contexts c..c+3; state %d MiB" % (
                    B * L.n_v_heads * L.d_k * L.d_v * 4 >> 20)}

    # chunked prefill: 1024-token prompts from S = 0, 32 requests, both layers; the bf16
    # products run as tcgen05 MMAs (bf16 hi/lo parts, fp32 accumulation in TMEM),
    # reported against the bf16 tensor peak and HBM
    tf_peak, tf_src = tensor_peak_bf16()
    for L, tag in ((I.GATED_LAYER, "prefill_gated_B32_L1024"),
                   (I.GDN_LAYER, "prefill_gated_delta_B32_L1024")):
        B, Lp = 32, 1024
        pool = pool_for(L, B, 8, 1)
        req = np.arange(B, dtype=np.int32)
        prompt = tokens(L, (B, Lp), 30)
        o_buf = torch.empty(B, Lp, L.n_v_heads, L.d_v, dtype=torch.float32, device=dev)
        us = timed(lambda: pool.prefill(req, *prompt, o=o_buf), 5)
        e = _entry_bytes(L)
        nbytes = B * Lp * (e + L.n_qk_heads * L.d_k * 2 + L.n_v_heads * L.d_v * 4) \
            + 2 * B * L.n_v_heads * L.d_k * L.d_v * 4
        flops = prefill_flops(L, B * Lp)
        tflops = flops / us / 1e6
        out[tag] = {"us_per_call": us, "mtok_per_s": B * Lp / us, "tflops": tflops,
                    "tensor_frac": tflops / tf_peak, "tensor_peak_tflops": tf_peak,
                    "tensor_peak_source": tf_src, "gbs": nbytes / us / 1e3,
                    "frac": nbytes / us / 1e3 / peak, "bytes": nbytes, "flops": flops,
                    "note": "chunk 64, tcgen05 bf16 MMAs with hi/lo parts, TMEM accumulators; "
                            "algorithmic flops of the chunked form"}
        del o_buf, prompt
        checked_close(pool)
    return out


# --------------------------------------------------------------------------- GPU arm
def run_ours(args, rank, world, local_rank):
    import torch
    from kv_buffered_decoding_gb300 import kvb

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    w = WORKLOAD
    L = w.layer
    B, m, bs = w.batch, w.m, w.block_size
    cfg = kvb.make_config(kvb.KVB_GATED_DELTA, kvb.KVB_BF16, L.n_qk_heads, L.n_v_heads, L.d_k,
                          L.d_v, m, bs, B, B, B, 1)
    pool = kvb.Pool(cfg, device=dev)
    gen = torch.Generator(device=dev)
    gen.manual_seed(1000 + rank)
    pool.state.normal_(0.0, 1.0 / np.sqrt(L.d_k), generator=gen)
    perm = np.random.default_rng(7 + rank).permutation(B)
    for r in range(B):
        pool.set_request(r, r, [int(perm[r])])
    rng = np.random.default_rng(w.seed + rank)
    bank_np = [I.draw_tokens(rng, L, (B,)) for _ in range(N_BANK)]

    def to_dev(tok):
        return (torch.from_numpy(tok["q"]).to(torch.bfloat16).to(dev),
                torch.from_numpy(tok["k"]).to(torch.bfloat16).to(dev),
                torch.from_numpy(tok["v"]).to(torch.bfloat16).to(dev),
                torch.from_numpy(tok["log_g"]).to(dev), torch.from_numpy(tok["beta"]).to(dev))

    bank = [to_dev(t) for t in bank_np]
    o = torch.empty(B, L.n_v_heads, L.d_v, dtype=torch.float32, device=dev)
    req = np.arange(B, dtype=np.int32)
    # staggered start: request r holds r mod m tokens
    occ = req % m
    for s in range(m - 1):
        rows = np.nonzero(occ > s)[0].astype(np.int32)
        sel = torch.from_numpy(rows).long().to(dev)
        pool.decode(rows, *[x.index_select(0, sel) for x in bank[s % N_BANK]])
    torch.cuda.synchronize()
    assert np.array_equal(pool.get_lengths()[:B], occ)

    for i in range(args.warmup):
        pool.decode(req, *bank[i % N_BANK], o=o)
    torch.cuda.synchronize()

    # algorithmic bytes of each timed step, from the host's exact length model
    lengths = pool.get_lengths()[:B].astype(np.int64)
    total_bytes, lens = 0, lengths.copy()
    for _ in range(args.steps):
        total_bytes += step_bytes(w, lens)
        lens = lens + 1
        lens[lens >= m] = 0

    stream = torch.cuda.current_stream(dev)
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local_rank) as clocks:
        start.record(stream)
        for i in range(args.steps):
            pool.decode(req, *bank[i % N_BANK], o=o)  # one kernel launch per step
        stop.record(stream)
        torch.cuda.synchronize()
    elapsed_ms = start.elapsed_time(stop)
    # the timed region is K back-to-back launches of the decode kernel on this stream
    launch_ms = [elapsed_ms / args.steps]
    clk = clocks.summary()
    elapsed_ms = max_over_ranks(elapsed_ms, dist)
    err = pool.get_error()
    if err is not None:
        raise RuntimeError(f"device error during bench: {err}")

    value = job_rate(world, B, args.steps, elapsed_ms)
    mean_launch_s = statistics.mean(launch_ms) / 1e3
    bytes_per_launch = total_bytes / args.steps
    achieved = bytes_per_launch / mean_launch_s / 1e9
    peak, peak_src = hbm_peak()

    # the same step end to end through the public API: every step's inputs are copied
    # in from pinned host memory and its output copied back, inside the timed region.
    # Two staging sets and separate copy streams let step i+1's upload and step i-1's
    # download overlap step i's kernel, as a serving loop would.
    host_bank = []
    for tok in bank_np:
        hb = []
        for key in ("q", "k", "v"):
            hb.append(torch.from_numpy(tok[key]).to(torch.bfloat16).pin_memory())
        for key in ("log_g", "beta"):
            hb.append(torch.from_numpy(tok[key]).pin_memory())
        host_bank.append(hb)
    stage = [[torch.empty_like(x, device=dev) for x in host_bank[0]] for _ in range(2)]
    o_dev = [torch.empty(B, L.n_v_heads, L.d_v, dtype=torch.float32, device=dev) for _ in range(2)]
    o_host = [torch.empty(B, L.n_v_heads, L.d_v, dtype=torch.float32).pin_memory() for _ in range(2)]
    h2d = sum(x.numel() * x.element_size() for x in host_bank[0])
    d2h = o_host[0].numel() * o_host[0].element_size()
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sync_ev = {key: [torch.cuda.Event() for _ in range(2)] for key in ("in", "run", "out")}

    def e2e_step(i):
        k = i % 2
        with torch.cuda.stream(up):
            if i >= 2:
                up.wait_event(sync_ev["run"][k])  # step i-2's kernel is done reading stage k
            for s_, h_ in zip(stage[k], host_bank[i % N_BANK]):
                s_.copy_(h_, non_blocking=True)
            sync_ev["in"][k].record(up)
        stream.wait_event(sync_ev["in"][k])
        if i >= 2:
            stream.wait_event(sync_ev["out"][k])  # step i-2's output has left o_dev[k]
        pool.decode(req, *stage[k], o=o_dev[k])
        sync_ev["run"][k].record(stream)
        with torch.cuda.stream(down):
            down.wait_event(sync_ev["run"][k])
            o_host[k].copy_(o_dev[k], non_blocking=True)
            sync_ev["out"][k].record(down)

    e2e_steps = args.steps
    for i in range(min(args.warmup, 8)):
        e2e_step(i)
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    s2, e2 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s2.record(stream)
    for i in range(e2e_steps):
        e2e_step(i)
    stream.wait_event(sync_ev["out"][(e2e_steps - 1) % 2])
    stream.wait_event(sync_ev["out"][e2e_steps % 2])
    e2.record(stream)
    torch.cuda.synchronize()
    e2e_ms = s2.elapsed_time(e2)
    e2e_ms = max_over_ranks(e2e_ms, dist)
    e2e_value = job_rate(world, B, e2e_steps, e2e_ms)

    # in-run HBM copy probe (1 GiB each way), best of 10
    src = torch.empty(1 << 28, dtype=torch.float32, device=dev).normal_(generator=gen)
    dst = torch.empty_like(src)
    probe = []
    for _ in range(12):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        kvb.copy_probe(src, dst)
        b_.record(stream)
        torch.cuda.synchronize()
        probe.append(a.elapsed_time(b_))
    copy_gbs = 2 * src.numel() * 4 / (min(probe[2:]) / 1e3) / 1e9
    tcopy = []
    for _ in range(12):
        a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        dst.copy_(src)
        b_.record(stream)
        torch.cuda.synchronize()
        tcopy.append(a.elapsed_time(b_))
    torch_copy_gbs = 2 * src.numel() * 4 / (min(tcopy[2:]) / 1e3) / 1e9
    del src, dst

    # recurrent decoding (m = 0) on the same workload, for the speed-up the method claims
    cfg0 = kvb.make_config(kvb.KVB_GATED_DELTA, kvb.KVB_BF16, L.n_qk_heads, L.n_v_heads, L.d_k,
                           L.d_v, 0, bs, 1, B, B, 1)
    pool0 = kvb.Pool(cfg0, device=dev)
    pool0.state.copy_(pool.state)
    for r in range(B):
        pool0.set_request(r, r, [])
    n_rec = max(16, min(args.steps, 512))
    for i in range(4):
        pool0.decode(req, *bank[i % N_BANK], o=o)
    torch.cuda.synchronize()
    a, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for i in range(n_rec):
        pool0.decode(req, *bank[i % N_BANK], o=o)
    b_.record(stream)
    torch.cuda.synchronize()
    rec_ms = a.elapsed_time(b_) / n_rec

    paths = None
    if world == 1 and not args.no_paths:
        del pool0
        paths = measure_paths(kvb, torch, dev, peak)

    if rank != 0:
        return
    cpu = None
    if world == 1 and not args.no_cpu_baseline:
        rate, steps, el = oracle_rate(w, args.cpu_seconds)
        all_rate, cores, tokens, all_el = oracle_rate_all_cores(args.cpu_seconds)
        cpu = {"value": all_rate, "unit": "tok/s", "cores": cores, "kind": "oracle",
               "sample": f"{cores} processes (one per host core), each 8 requests x 32 heads "
                         f"of consecutive decode steps for {args.cpu_seconds:.0f} s ({tokens} "
                         "tokens in all), fp64 per-token recurrence (numpy, one thread each)",
               "one_core": {"value": rate, "cores": 1,
                            "sample": f"8 requests x 32 heads, {steps} consecutive decode "
                                      f"steps ({el:.1f} s), one process"}}
    line = {
        "metric": METRIC, "value": value, "unit": "tok/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 KV / f32 state",
        "data": "synthetic (seeded; state iid normal, q/k L2-normalised, beta = sigmoid(N), "
                "log-decay = -0.1 softplus(N))",
        "config": workload_config(),
        "hbm_gbs": achieved,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": ncu_traffic(),
                     "kernel": "decode_stream_kernel<bf16, gated_delta> (persistent, d=128)",
                     "algorithmic_bytes_per_launch": bytes_per_launch,
                     "mean_launch_us": mean_launch_s * 1e6, "peak_source": peak_src},
        "copy_probe_gbs": copy_gbs,
        "torch_copy_gbs": torch_copy_gbs,
        "frac_of_copy_probe": achieved / copy_gbs,
        "recurrent_m0_ms_per_step": rec_ms,
        "speedup_vs_recurrent": rec_ms / (elapsed_ms / args.steps),
        "e2e": {"value": e2e_value, "unit": "tok/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "gpu_launches": args.steps,
        "clocks": clk,
        "cpu_baseline": cpu,
        "paths": paths,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=4096)
    ap.add_argument("--warmup", type=int, default=32)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-paths", action="store_true", help="skip the verify/flush/short timings")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
    if args.impl == "reference":
        run_reference(args, rank, world)
    else:
        from kv_buffered_decoding_gb300 import build as _build
        if rank == 0 or world == 1:
            _build.build()
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        run_ours(args, rank, world, local_rank)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
