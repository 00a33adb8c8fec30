"""The fp64 oracle over many independent requests, in worker processes.

Requests never interact, so the parity tests of the full-size workloads split
them into chunks and run the oracle (unchanged) on every chunk in a pool of
worker processes.  The pool uses the ``spawn`` start method: a process forked
after CUDA has been initialised in the parent would hang.  Workers import only
numpy and the oracle; they compare the GPU results they are given with the
oracle's and return per-tensor errors, so no large array travels back.

Error metric (per tensor): max_i |x_i - r_i| / max_i |r_i| over one output o_t
of one request (all its value heads) or over one request's state.
"""
from __future__ import annotations

import multiprocessing as mp
import os

import numpy as np


def rel_err_rows(x, ref, nlead: int) -> np.ndarray:
    """Normwise relative error of every tensor indexed by the first ``nlead`` axes."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert x.shape == r.shape, (x.shape, r.shape)
    axes = tuple(range(nlead, r.ndim))
    num = np.abs(x - r).max(axis=axes)
    den = np.maximum(np.abs(r).max(axis=axes), 1e-30)
    return num / den


def workers() -> int:
    try:
        n = len(os.sched_getaffinity(0))
    except AttributeError:
        n = os.cpu_count() or 1
    return max(1, min(16, n))


def run(fn, tasks):
    """fn(task) for every task, in a spawn pool; results in task order."""
    tasks = list(tasks)
    if len(tasks) == 1:
        return [fn(tasks[0])]
    from concurrent.futures import ProcessPoolExecutor
    # a worker that dies raises BrokenProcessPool instead of being restarted
    with ProcessPoolExecutor(min(workers(), len(tasks)), mp_context=mp.get_context("spawn")) as ex:
        return list(ex.map(fn, tasks))


def chunks(n: int, size: int):
    return [np.arange(i, min(n, i + size)) for i in range(0, n, size)]


# ----------------------------------------------------------------- worker tasks
def decode_errors(task):
    """Errors of one chunk of requests decoding the same steps.

    task: dict with S0 [r, Hv, dk, dv]; hist: token dict laid out [T, r, ...]
    (each request's whole history, warm-up tokens first, already aligned so
    that every request has the same length T); out [steps, r, Hv, dv] = GPU
    outputs of the last ``steps`` tokens (earlier outputs are not compared); state [r, Hv, dk, dv] = GPU states, compared
    with the oracle state after token index fold_at[r] (-1: the initial state);
    variant, scale.
    Returns (worst output error per request, state error per request).
    """
    import oracle
    S0 = task["S0"]
    hist = task["hist"]
    T = hist["v"].shape[0]
    steps = task["out"].shape[0]
    fold_at = task["fold_at"]
    keep = sorted({int(t) for t in fold_at if t >= 0})
    o_ref, _, states = oracle.decode_sequence(S0, hist, task["variant"], task.get("scale", 1.0),
                                              keep_states=keep)
    err_o = rel_err_rows(task["out"], o_ref[T - steps:], 2).max(axis=0)
    err_s = np.empty(len(fold_at))
    for i, t in enumerate(fold_at):
        ref = S0[i] if t < 0 else states[int(t)][i]
        err_s[i] = rel_err_rows(task["state"][i][None], ref[None], 1)[0]
    return err_o, err_s


def verify_errors(task):
    """Errors of one chunk of requests over every verify + accept round.

    task: S0 [r, Hv, dk, dv]; drafts: token dict laid out [rounds, T, r, ...];
    acc [rounds, r] accepted prefix lengths; out [rounds, r, T, Hv, dv] GPU
    outputs; checkpoints: {round: GPU states [r, ...] after that round};
    fold_rounds [rounds, r] bool (the request folded in that round); final:
    GPU states after a closing flush; variant, scale.
    Returns (worst output error per request, worst checkpoint state error per
    request, final state error per request).
    """
    import oracle
    S_hist = task["S0"].astype(np.float64)
    drafts, acc = task["drafts"], task["acc"]
    rounds = acc.shape[0]
    n_r = S_hist.shape[0]
    S_fold = S_hist.copy()  # the state the pool holds: the one at each request's last fold
    err_o = np.zeros(n_r)
    err_ck = np.zeros(n_r)
    ck = task["checkpoints"]
    for rnd in range(rounds):
        d = {key: (None if val is None else val[rnd]) for key, val in drafts.items()}
        T = d["v"].shape[0]
        o_ref, _, states = oracle.decode_sequence(S_hist, d, task["variant"], task.get("scale", 1.0),
                                                  keep_states=range(T))
        got = np.swapaxes(task["out"][rnd], 0, 1)  # [T, r, Hv, dv]
        err_o = np.maximum(err_o, rel_err_rows(got, o_ref, 2).max(axis=0))
        for i in range(n_r):
            j = int(acc[rnd, i])
            if j > 0:
                S_hist[i] = states[j - 1][i]
        folded = task["fold_rounds"][rnd]
        S_fold[folded] = S_hist[folded]
        if rnd in ck:
            err_ck = np.maximum(err_ck, rel_err_rows(ck[rnd], S_fold, 1))
    err_final = rel_err_rows(task["final"], S_hist, 1)
    return err_o, err_ck, err_final


def short_errors(task):
    """Errors of short-context incarnations: each is the recurrence from S = 0.

    task: items = list of (history token dict [T, Hv|Hk, d], GPU outputs [T, Hv, dv]);
    variant, d_k, d_v, scale.  Returns the worst output error per item.
    """
    import oracle
    out = []
    for hist, got in task["items"]:
        o_ref = oracle.short_context(hist, task["variant"], task["d_k"], task["d_v"],
                                     task.get("scale", 1.0))
        out.append(rel_err_rows(got, o_ref, 1).max())
    return np.array(out)
