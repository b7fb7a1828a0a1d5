"""The benchmark's work accounting (the algorithmic FLOPs and bytes its
roofline divides by) against the oracle and against hand counts.

bench.py keeps its own copy of the data-independent growth schedule to count
state rows per query; these tests tie it to the pinned oracle's slot counts,
and the per-query key counts to a direct enumeration of the window rule
("Key-Value Means", gist.science technical summary, Core mechanisms 1 and 3).
"""
import numpy as np
import pytest

import bench
import oracle
from compressed_kv_state_gb300 import workloads as wl

CASES = [
    wl.Workload("acc_fixed", B=1, H=1, N=700, chunk=32, window=64, n_sinks=4, max_slots=20),
    wl.Workload("acc_sqrt", B=1, H=1, N=900, chunk=32, window=64, n_sinks=8, sched=1,
                max_slots=200),
    wl.Workload("acc_pow", B=1, H=1, N=1100, chunk=64, window=128, n_sinks=16, sched=1,
                max_slots=400, coef=2.0, expo=0.75),
]


def _oracle_slots_after_each_event(w):
    """Slot count after every fold event, read off the oracle's per-token kinds."""
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((3, 1, w.N, w.d))
    g = np.full((1, w.N), 0.5)
    cfg = oracle.OracleConfig(head_dim=w.d, rope_dims=w.rope_dims, chunk=w.chunk, window=w.window,
                              n_sinks=w.n_sinks, sched=w.sched, max_slots=w.max_slots,
                              coef=w.coef, expo=w.expo)
    _, st, dbg = oracle.prefill(cfg, q, k, v, g, threads=1)
    new_slots = (dbg["kind"][0] != oracle.MERGED).sum(axis=1)  # appended + sink founders
    return np.cumsum(new_slots), st[0].n


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_schedule_matches_oracle(w):
    n_after, n_final = _oracle_slots_after_each_event(w)
    sched = bench._schedule(w)
    assert list(sched) == n_after.tolist()
    assert (sched[-1] if sched else 0) == n_final


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_key_counts_by_enumeration(w):
    """Per query: the state rows of the events before its chunk's window, and
    every token from the window's first chunk up to the query itself."""
    n_after, _ = _oracle_slots_after_each_event(w)
    C, Wc = w.chunk, w.window // w.chunk
    state_pairs = win_pairs = 0
    for p in range(w.N):
        c = p // C
        folded = [e for e in range(len(n_after)) if e + Wc + 1 <= c]
        state_pairs += int(n_after[folded[-1]]) if folded else 0
        visible = [t for t in range(p + 1) if t // C >= c - Wc]
        win_pairs += len(visible)
    aw = bench.attention_work(w)
    assert aw["state_pairs"] == state_pairs and aw["window_pairs"] == win_pairs
    d, r = w.d, w.rope_dims
    assert aw["flops"] == state_pairs * (2 * (d - r) + 2 * d) + win_pairs * 4 * d


def test_decode_bytes_by_parts():
    """One decode step, per (b, h) row: window keys and values (bf16) of the W + r + 1
    visible tokens, the state's read view (key on the non-rotary dims, value), the
    query and output, the new key and value written into the ring, and its gate."""
    dw = wl.Workload("dec", B=64, H=16, N=0, window=512, chunk=128, max_slots=512)
    d, r, n, rin = 64, 32, 512, 5
    per_row = ((512 + rin + 1) * (d + d) * 2      # window K and V
               + n * ((d - r) + d) * 2            # state view
               + (d + d) * 2                      # q, out
               + (d + d) * 2 + 4)                 # new k, v into the ring; gate
    assert bench.decode_bytes(dw, rin, n) == per_row * 64 * 16


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fold_flops_by_enumeration(w):
    """Similarity work of every fold event from the oracle's per-token kinds: each
    candidate (not a sink founder) against every mergeable slot that existed before
    the event, and each merged token against the slots the event appended."""
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal((3, 1, w.N, w.d))
    g = np.full((1, w.N), 0.5)
    cfg = oracle.OracleConfig(head_dim=w.d, rope_dims=w.rope_dims, chunk=w.chunk, window=w.window,
                              n_sinks=w.n_sinks, sched=w.sched, max_slots=w.max_slots,
                              coef=w.coef, expo=w.expo)
    _, _, dbg = oracle.prefill(cfg, q, k, v, g, threads=1)
    pairs, n = 0, 0
    for kinds in dbg["kind"][0]:
        sinks = int((kinds == oracle.SINK).sum())
        appended = int((kinds == oracle.APPENDED).sum())
        merged = int((kinds == oracle.MERGED).sum())
        mergeable_before = n + sinks - w.n_sinks
        pairs += (appended + merged) * max(0, mergeable_before) + merged * appended
        n += sinks + appended
    assert bench.fold_work(w) == 2 * w.d * pairs
